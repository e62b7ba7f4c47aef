"""GB300-native spatial-transformer sampling (placeholder; binding added with the library)."""
