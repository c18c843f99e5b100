"""NVFP4 paged-KV attention decode / extend for GB300 (sm_103a).

The compute path is the C-ABI library libnvfp4kv.so (include/nvfp4kv.h),
built in-tree by ``build.build()``; this package only marshals arguments.
"""
from .api import (NvFp4KvError, PagedCache, Plan, default_sm_scale,  # noqa: F401
                  nvfp4kv_decode_attend, nvfp4kv_decode_merge, nvfp4kv_decode_plan,
                  nvfp4kv_decode_run, nvfp4kv_merge_states, nvfp4kv_quantize_append,
                  nvfp4kv_workspace_flags, nvfp4kv_decode_run_static,
                  nvfp4kv_static_workspace_flags,
                  nvfp4kv_decode_append_run, nvfp4kv_dequantize_paged)
