"""GB300-native device-wide scan and stream compaction (placeholder; binding follows)."""
