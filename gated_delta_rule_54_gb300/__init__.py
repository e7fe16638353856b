"""GB300-native chunked gated delta rule with state/W fake QDQ (placeholder, filled below)."""
