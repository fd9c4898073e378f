"""libmsa: the decode hot path of MiniMax Sparse Attention (MSA) over an NVFP4
paged KV cache, as hand-written CUDA kernels for GB300 (sm_103a) behind a C ABI
(include/msa.h). This package holds the kernels (csrc/), the in-tree build, a
thin ctypes binding and the seeded synthetic-workload generator (synth/)."""
from . import _lib  # noqa: F401  (binding; loads libmsa.so on first call)
from .api import DecodeBatch, KVCache, MSADecoder, dequant_rows  # noqa: F401
from ._lib import MSAError  # noqa: F401
