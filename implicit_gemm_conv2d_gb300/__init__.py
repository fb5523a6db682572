"""Implicit-GEMM conv2d for GB300 (sm_103a): forward (+ fused ReLU, + optional
per-channel bias), data gradient, weight gradient and bias gradient of a
no-padding, square-kernel, strided NCHW convolution, as hand-written CUDA
kernels behind a C ABI (include/conv.h).

``binding`` holds the ctypes binding (names match the C entry points);
``synth`` the seeded synthetic inputs; ``build`` the nvcc build."""

from .binding import (ALGO_AUTO, ALGO_DIRECT, ALGO_FFMA, ALGO_TC, BF16, F32, OP_BWD_BIAS,  # noqa: F401
                      OP_BWD_DATA, OP_BWD_FILTER, OP_FWD, ConvDesc, ConvError, bwd_bias, bwd_data,
                      bwd_filter, conv_bwd_bias, conv_bwd_data, conv_bwd_filter,
                      conv_bwd_filter_workspace_size, conv_fwd, conv_fwd_bias, conv_query,
                      conv_query_for_device, conv_set_algo, fwd, make_desc, out_dims)
