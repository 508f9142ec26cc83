"""GB300-native Gated DeltaNet recurrence (placeholder; binding added with the C-ABI)."""
