"""GB300-native speculative-decoding verify sampler (placeholder; binding added with the library)."""
