"""GB300-native segmented (batched) top-k by multi-pass radix digit selection."""
