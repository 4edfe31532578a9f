"""Exact tiled attention (FlashAttention-style) for GB300 / sm_103a.

The compute path is the C-ABI library ``libfattn.so`` built from ``csrc/``;
``fattn`` is its thin Python binding (argument marshalling only). The library
is loaded lazily by ``fattn`` so that ``inputs`` can be imported on machines
without a GPU.
"""
