// bwd_tcgen05_d64_v128.cu -- the attention backward kernels of
// bwd_tcgen05.cu built for key head dim 64 and value head dim 128 (a
// translation unit of the same source).
#define ATTN_BWD_HEAD_DIM 64
#define ATTN_BWD_VALUE_DIM 128
#include "bwd_tcgen05.cu"
