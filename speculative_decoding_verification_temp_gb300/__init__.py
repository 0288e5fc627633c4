"""GB300-native speculative-sampling verification (placeholder, binding follows)."""
