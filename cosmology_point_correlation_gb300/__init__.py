"""GB300-native graph-based 3pCF / parity-4pCF counting (placeholder, filled in below)."""
