"""GB300-native tensor layout permutation (sm_103a)."""
