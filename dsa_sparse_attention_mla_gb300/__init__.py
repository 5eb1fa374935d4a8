"""GB300-native DSA sparse MLA attention (placeholder; binding added next)."""
