"""GB300-native DSA decode hot path (placeholder; the binding lands with the library)."""
