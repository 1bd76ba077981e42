"""GB300 (sm_103a) fused LM-head + exact Gumbel-max sampling.

The compute lives in libfs_sample.so (C ABI: include/fs_sample.h); this
package is its Python binding.  Build the library with ``build.build()``.
"""
from ._lib import (FS_DTYPE_BF16, FS_DTYPE_F32, FS_FLAG_NO_NOISE,  # noqa: F401
                   FS_STAGE1_MULTICAST_PAIR, FS_STAGE1_ONE_CTA, FS_STAGE1_PAIR_MMA, STAGE1_FORM_NAMES,
                   fs_stage1_form,
                   FS_FLAG_STORE_LOGITS, FSError, Transforms, fs_debug_gumbel, fs_debug_noise, fs_get_device_status,
                   fs_last_error_string, fs_logits_gemm, fs_plan_info, fs_release_workspaces,
                   fs_sample, fs_sample_ex, fs_sample_host, fs_sample_from_logits, fs_sample_logprob, fs_sample_noalloc, fs_sample_shard, fs_combine_groups,
                   fs_sample_transformed, fs_sample_unfused,
                   fs_stage1, fs_stage2, fs_version, fs_workspace_size, lib, workspace)
