"""GB300-native paged split-K decode attention (libpdecode) and its Python binding."""
