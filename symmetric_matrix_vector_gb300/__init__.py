"""GB300-native xSYMV / xHEMV (placeholder; binding added with the CUDA library)."""
