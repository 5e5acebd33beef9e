"""GB300-native (sm_103a) blocked GQA flash attention.

``binding`` exposes the C entry points of libfa_gb300.so (fa_fwd, fa_bwd, ...)
through ctypes; ``inputs`` builds the seeded synthetic workloads.  Importing the
package loads nothing: the library is loaded on first use and every call fails
loudly when it is missing.
"""
__all__ = ["binding", "inputs", "build"]
