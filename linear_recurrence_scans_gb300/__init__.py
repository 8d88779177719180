"""GB300-native minGRU scan library (placeholder; the binding follows)."""
