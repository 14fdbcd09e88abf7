"""BMMC index permutations on GB300 (placeholder; binding added with the library)."""
