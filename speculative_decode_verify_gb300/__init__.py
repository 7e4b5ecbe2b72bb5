"""GB300-native speculative-decoding verify attention (placeholder; binding added next)."""
