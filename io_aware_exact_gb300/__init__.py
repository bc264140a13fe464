"""GB300-native exact IO-aware attention (placeholder; binding follows)."""
