"""GB300-native dense point-cloud neighbor search (FPS, kNN, Ball Query)."""
