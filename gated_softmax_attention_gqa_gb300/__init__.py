"""GB300-native gated softmax attention with GQA (libgattn)."""
