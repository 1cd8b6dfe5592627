"""The library's compiled configuration names, for parametrising tests at
collection time. The library is host code plus device images: it builds and
loads without a GPU, and its configuration table is host data."""
_NAMES = None


def compiled_config_names():
    global _NAMES
    if _NAMES is None:
        from dense_fp16_gemm_02_gb300 import build, wgemm
        build.build()
        _NAMES = wgemm.config_names()
    return _NAMES


def plain_fp32():
    """Plain (not fused) configurations writing fp32 C."""
    return [n for n in compiled_config_names() if not n.endswith("_h") and "_ab" not in n]


def plain_16bit():
    """Plain (not fused) configurations writing a 16-bit C."""
    return [n for n in compiled_config_names() if n.endswith("_h") and "_ab" not in n]
