"""GB300-native MLA KV prolog: a C-ABI CUDA library and its Python binding."""
