"""libmoeroute: MoE expert-routing statistics for locality-aware serving on GB300.

The compute lives in the C ABI library (`include/moeroute.h`, CUDA kernels
for sm_103a under `csrc/`); this package only builds it (`build.py`) and
binds it (`_native.py`, ctypes, same names as the C entry points).
`pipeline.py` strings the entry points into the routing-statistics step
that the tests and the bench run.
"""
from ._native import (moer_dims, make_dims, MoerError, moer_workspace_bytes,  # noqa: F401
                      moer_topk_signature, moer_topk_signature_noalloc, moer_block_stitch, moer_affinity_load, moer_route,
                      moer_idf_fit, moer_gate_workspace_bytes, moer_gate_topk, moer_ids_signature, moer_ws_status, moer_status_str, moer_version, moer_set_extent_checks,
                      moer_extent_checks, moer_buffer_holds, EXPORTS)
