"""GB300-native paged-KV attention: the binding lives in ``_binding``."""
