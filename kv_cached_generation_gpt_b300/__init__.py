"""B300-native KV-cached GPT-2 generation (sm_103a)."""
