"""GB300 (sm_103a) single-query decode attention: dense, paged and sparse.

The compute lives in hand-written CUDA kernels behind a C ABI (``include/decode_attn.h``,
``libdecode_attn.so``); :mod:`.binding` marshals torch tensors into those calls.  Importing
this package does not load the library; the first call does, and raises if it was not built.
"""
_BINDING_NAMES = (
    "DecodeAttnError", "abi_version", "decode_attn_dense", "decode_attn_paged",
    "decode_attn_sparse", "decode_attn_workspace_size", "decode_attn_workspace_init",
    "decode_attn_set_grid_limit", "decode_attn_read_device_error", "library_path",
    "load_library", "new_workspace", "run_case", "decode_attn_append_paged",
    "decode_attn_append_ring", "decode_attn_dense_device_len", "decode_attn_dense_mq",
    "decode_attn_paged_mq", "decode_attn_check_wait_timeout", "decode_attn_spec_check",
    "decode_attn_dense_spec", "decode_attn_dense_noalloc", "decode_attn_status_string",
    "decode_attn_abi_version", "DecodeAttnSpec",
    "DA_VARIANT_DENSE", "DA_VARIANT_PAGED", "DA_VARIANT_SPARSE",
)


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
