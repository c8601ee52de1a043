"""GB300 (sm_103a) MLA paged-KV decode.

The decode runs in ``libmla_decode.so`` (hand-written CUDA for sm_103a behind
the C ABI in ``include/mla_decode.h``).  ``_lib`` is the ctypes binding (same
names as the C entry points), ``api`` adds torch buffer plumbing, and ``synth``
draws seeded synthetic inputs.  Importing the package loads nothing; the
library is loaded on first use and a missing library is an error.
"""
