"""ctypes binding of librf.so (placeholder until the C-ABI lands)."""


def load():
    raise RuntimeError("librf.so not built")
