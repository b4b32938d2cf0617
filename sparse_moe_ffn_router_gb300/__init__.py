"""GB300-native sparse Mixture-of-Experts feed-forward layer (placeholder, filled below)."""
