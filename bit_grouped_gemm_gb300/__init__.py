"""GB300 (sm_103a) W4A16 mixture-of-experts block.

The compute lives in ``libmoe_w4.so`` (C ABI in ``include/moe_w4.h``);
``binding`` marshals arguments to it and ``synth`` draws the seeded synthetic
workloads. Importing the package does not load the library; the first call
does, and raises if the library has not been built.
"""
from .binding import (KERNEL_KINDS, MoeError, MoeExperts, MoeLayer, MoePlanDesc, MoeRouting, MoeW4,  # noqa: F401
                      experts, load_library, moe_debug_wait_timeout, moe_enable_timing, moe_debug_buffer,
                      moe_forward_layer, moe_forward_stack, moe_layers, moe_get_error, moe_grouped_w4_ffn, moe_last_gemm_path,
                      moe_plan_create, moe_plan_destroy, moe_plan_scratch_bytes,
                      moe_read_timing, moe_residual_add, moe_route, moe_route_noalloc, moe_set_tail_split,
                      moe_status_string,
                      moe_version, plan_desc)
