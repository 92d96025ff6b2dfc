"""The debug build compiles and exports the same boundary (CPU only)."""
import ctypes

from rmsnorm_fwd_bwd_gb300 import binding as B
from rmsnorm_fwd_bwd_gb300 import build as build_mod


def test_debug_build_links_and_exports_every_symbol():
    lib = ctypes.CDLL(build_mod.build(debug=True))
    for name in B.header_functions():
        assert hasattr(lib, name), name
