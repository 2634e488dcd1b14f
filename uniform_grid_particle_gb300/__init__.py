"""GB300-native uniform spatial grid build (count -> scan -> scatter -> gather)."""
