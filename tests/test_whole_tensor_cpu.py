"""Host logic of the whole-tensor comparison: the blocks cover every (b, h)
sequence exactly once, and the block-by-block sums give the same relative
Frobenius error as one comparison over the whole tensor."""
import numpy as np
import torch

from tests.pins import rel
from tests.whole_tensor import head_blocks, whole_errors


def test_blocks_cover_every_sequence_once():
    for B, T, H, width, budget in [(3, 100, 7, 64, 100 * 64 * 8 * 3), (1, 10, 5, 8, 1),
                                   (2, 5, 4, 16, 1 << 30)]:
        seen = []
        for b, h0, h1 in head_blocks(B, T, H, width, budget):
            assert 0 <= b < B and 0 <= h0 < h1 <= H
            assert (h1 - h0) * T * width * 8 <= max(budget, T * width * 8)
            seen += [(b, h) for h in range(h0, h1)]
        assert sorted(seen) == [(b, h) for b in range(B) for h in range(H)]


def test_blockwise_error_equals_whole_error():
    gen = torch.Generator().manual_seed(3)
    B, T, H, K, V = 2, 9, 5, 4, 3
    x = {"q": torch.randn(B, T, H, K, generator=gen), "k": torch.randn(B, T, H, K, generator=gen),
         "v": torch.randn(B, T, H, V, generator=gen), "g": torch.randn(B, T, H, generator=gen),
         "beta": torch.rand(B, T, H, generator=gen), "h0": torch.randn(B, H, K, V, generator=gen)}
    # a stand-in "oracle" that is a fixed function of each sequence's own inputs
    f_o = lambda s: (s["v"].double() * 2 + s["g"].double()[..., None]).numpy()
    f_h = lambda s: (s["h0"].double() * 3).numpy()
    ref_o = f_o(x)
    ref_h = f_h(x)
    got_o = torch.from_numpy(ref_o + 0.01 * np.cos(np.arange(ref_o.size)).reshape(ref_o.shape))
    got_h = torch.from_numpy(ref_h + 0.02 * np.sin(np.arange(ref_h.size)).reshape(ref_h.shape))
    eo, eh = whole_errors(x, got_o, got_h, lambda s: (f_o(s), f_h(s)), budget=T * K * 8)
    assert abs(eo - rel(got_o.numpy(), ref_o)) < 1e-12
    assert abs(eh - rel(got_h.numpy(), ref_h)) < 1e-12
