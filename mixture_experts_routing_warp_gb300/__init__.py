"""GB300-native Mixture-of-Experts layer forward (placeholder; binding follows)."""
