"""GB300-native Kimi Delta Attention (KDA) recurrent decode."""
