"""The pins are discriminating: plausible mistakes planted in a copy of the C
oracle (on the CPU, in a temporary directory) must each fail at least one pin."""
import pytest

from oracle import recurrence
from tests import pins

MUTANTS = {
    "no_decay": ("S[e] *= a;", "S[e] *= 1.0;"),
    "g_read_as_per_token": ("gt - j->g[row - H]", "gt"),
    "previous_token_index": ("gt - j->g[row - H]", "gt - j->g[row - 1]"),
    "chunk_start_off_by_one": ("(t % j->chunk == 0) ? gt", "(t % j->chunk == 1) ? gt"),
    "beta_dropped": ("d[c] = bt * (vt[c] - r);", "d[c] = (vt[c] - r);"),
    "read_sign": ("d[c] = bt * (vt[c] - r);", "d[c] = bt * (vt[c] + r);"),
    "scale_dropped": ("ot[c] = j->scale * r;", "ot[c] = r;"),
    "query_with_key": ("r += S[(size_t)i * V + c] * qt[i];", "r += S[(size_t)i * V + c] * kt[i];"),
    "write_without_key": ("Si[c] += kt[i] * d[c];", "Si[c] += d[c];"),
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = recurrence.SRC.read_text()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mut = tmp_path / "mutant.c"
    mut.write_text(src.replace(old, new))
    lib = recurrence.load(recurrence.build(force=True, src=mut, out=tmp_path / "libmutant.so"))

    def fwd(q, k, v, g, beta, scale, h0, chunk):
        return recurrence.forward(q, k, v, g, beta, scale, h0, chunk=chunk, nthreads=1, lib=lib)

    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(fwd)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"
