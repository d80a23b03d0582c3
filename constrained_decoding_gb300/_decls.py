"""ctypes signatures of the library entry points beyond the GEMM test entry."""


def declare(lib, sig):
    return None
