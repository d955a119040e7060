"""GB300-native fused MoE layer with per-request LoRA adapters (sm_103a).

The compute path is the C-ABI library libmoe_lora.so (CUDA kernels for sm_103a);
`expert_gemm_gb300.moe_lora` is its thin ctypes binding.  Importing the package
loads nothing; the binding loads the library on first use and raises if it is
missing.
"""
__all__ = ["moe_lora", "workloads"]
