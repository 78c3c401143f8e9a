"""GB300-native Gated DeltaNet recurrence (placeholder until the binding lands)."""
