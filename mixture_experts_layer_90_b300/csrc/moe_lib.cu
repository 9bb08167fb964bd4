// Single translation unit of the CUDA library: the device status word and
// every kernel live in one module, so one copy of the status word is seen by
// all kernels and by moe_get_device_status.
#include "abi.cu"
#include "backward.cu"
#include "balance.cu"
#include "combine.cu"
#include "gemm.cu"
#include "permute.cu"
#include "permute_static.cu"
#include "quant.cu"
#include "route.cu"
#include "train.cu"
