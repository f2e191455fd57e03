"""B300-native N:M sparse matrix-vector product for LLM decoding.

The compute path is libnm.so (hand-written CUDA for sm_103a, C ABI in
include/nm.h); ``sparse_spmv_memory_02_b300.nm`` is its thin Python binding.
"""
from .nm import (NM_F16, NM_F32, NM_MAX_BATCH, NM_MAX_BATCH_TC, NMError, PackedMatrix, lib, nm_last_error,  # noqa: F401
                 nm_calib_accumulate, nm_device_errors, nm_pack, nm_packed_sizes, nm_prune_pack, nm_select_mask, nm_spmv, nm_spmv_batched, nm_spmv_gate_up_silu, nm_spmv_group, nm_status_str, nm_unpack,
                 nm_version)
