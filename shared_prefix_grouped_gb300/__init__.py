"""GB300-native grouped attention for shared-prefix (Prefix Grouper) workloads."""
