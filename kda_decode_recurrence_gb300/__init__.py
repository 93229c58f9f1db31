"""GB300-native KDA decode recurrence and fused KDA block (placeholder)."""
