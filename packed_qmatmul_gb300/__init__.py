"""GB300-native weight-only quantized products over packed block formats."""
