"""MoDA (Mixture-of-Depths Attention) forward on GB300 (sm_103a).

Thin Python face of the C-ABI library ``libmoda.so`` (declared in
``include/moda.h``): argument marshalling only, every step of the path runs in
the library's CUDA kernels. The library is loaded on first use and its absence
is an error; there is no CPU fallback.
"""
from .binding import (MODA_OK, ModaError, library_path, load, moda_bwd, moda_bwd_noalloc,
                      moda_decode, moda_decode_workspace_bytes, moda_depth_cache_admit,
                      moda_depth_mass, moda_depth_mass_workspace_bytes, moda_depth_write,
                      moda_depth_write_at, moda_fwd, moda_fwd_host_workspace_bytes,
                      moda_fwd_layer_major, moda_fwd_layer_major_host, moda_get_device_error,
                      moda_kv_proj_write, moda_pack_depth, moda_selftest_wait_timeout,
                      moda_status_string)

__all__ = ["MODA_OK", "ModaError", "library_path", "load", "moda_bwd", "moda_bwd_noalloc",
           "moda_decode", "moda_decode_workspace_bytes", "moda_depth_cache_admit",
           "moda_depth_mass", "moda_depth_mass_workspace_bytes", "moda_depth_write",
           "moda_depth_write_at", "moda_fwd", "moda_fwd_host_workspace_bytes",
           "moda_fwd_layer_major", "moda_fwd_layer_major_host", "moda_get_device_error",
           "moda_kv_proj_write", "moda_pack_depth", "moda_selftest_wait_timeout",
           "moda_status_string"]
