"""GB300 (sm_103a) block-quantized decode: Q8_0 activation quantiser,
M = 1 Q4_0 / Q8_0 matrix-vector products and the small-M batched product,
Q4_K-style super-block products (per-256 quantiser, integer-domain scales),
block-128 / float16-scale / signed-offset 8-bit products,
the decode steps around them (rmsnorm, RoPE, GQA attention, silu_mul, add),
behind the C ABI of libmlq.so (include/mlq.h).

The Python names below are the C entry points of the same names; they only
marshal arguments (see binding.py).
"""
from .binding import (  # noqa: F401
    EXPORTS, LIB_PATH, ChainCall, ChainPhase, ChainProduct, mlq_chain_workspace_bytes,
    mlq_decode_chain, mlq_decode_chain_static, FusedCall, mlq_matvec_fused, PhaseCall, PhaseProduct, mlq_decode_phase, MLQ_E_ALIGN, MLQ_E_ARCH, MLQ_E_CUDA, MLQ_E_NULL, MLQ_E_SHAPE,
    MLQ_E_TIMEOUT, MLQ_E_BOUNDS, MLQ_E_TYPE, MLQ_MAX_COLS, MLQ_MAX_M, MLQ_OK, MLQ_Q4_0, MLQ_Q8_0, MLQ_QK,
    MLQ_F_STATIC_WEIGHTS, MLQ_F_STATIC_INPUT, MlqError, QAct, QTensor, lib, mlq_block_sumi, mlq_debug_set_wait_limit_ns,
    mlq_gemm_q4_small_m, mlq_init, mlq_last_device_error, mlq_matvec_q4, mlq_matvec_q8,
    mlq_prefetch_l2, mlq_quantize_q8, mlq_status_str,
    MLQ_MAX_SEQ, MLQ_MAX_HEAD_DIM, mlq_rmsnorm, mlq_add_rmsnorm, mlq_add, mlq_softmax, mlq_silu_mul,
    mlq_rope_tables, mlq_rope, mlq_attention,
    MLQ_QKK, Q4KTensor, Q8KAct, mlq_quantize_q8k, mlq_matvec_q4k, mlq_block_sums_q4k, mlq_q4k_phase,
    NBitsTensor, BlkAct, mlq_quantize_blk, mlq_matvec_nbits, mlq_block_sumi_nbits, mlq_nbits_phase,
)
