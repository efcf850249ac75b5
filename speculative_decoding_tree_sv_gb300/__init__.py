"""GB300-native verification of speculative-decoding draft trees.

The compute path is a C-ABI CUDA library (``libsv.so``, sources in
``csrc/``, declarations in ``include/sv.h``) built for sm_103a.  The Python
side only marshals arguments: ``binding`` exposes ``sv_tree_attention``,
``sv_greedy_accept`` and ``sv_kv_commit`` under the same names as the C
entry points.  The library is loaded on first use and a missing build raises
an error; there is no fallback.
"""

__all__ = ["cost"]
