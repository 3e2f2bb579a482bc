"""GB300-native chunked forward of the gated delta rule (Gated DeltaNet)."""
