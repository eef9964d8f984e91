"""GB300-native fused AdamW step with Philox-keyed stochastic rounding to bf16.

The computation lives in ``libasr.so`` (CUDA kernels for sm_103a behind a C
ABI, declared in ``include/asr.h``); this package is its ctypes binding plus
the synthetic workload definitions used to exercise it.
"""
from ._lib import (  # noqa: F401
    ASR_BF16, ASR_F32, ASR_ROUND_RNE, ASR_ROUND_SR, AsrError, asr_adamw_prepare,
    asr_adamw_sr_multi_tensor, asr_adamw_sr_multi_tensor_static, asr_adamw_sr_step,
    asr_gemm_bf16_sr, asr_last_cuda_error, asr_philox4x32, asr_status_string,
    asr_stochastic_round_bf16, asr_take_device_error, asr_take_device_error_async, asr_selftest_wait_timeout,
    asr_kernel_launches, asr_adamw_sr_multi_tensor_host, lib, make_host_table, make_table,
)
from .optim import AdamWSR, DeviceError  # noqa: F401,E402
