// bwd_tcgen05_d128_v64.cu -- the attention backward kernels of
// bwd_tcgen05.cu built for key head dim 128 and value head dim 64 (a
// translation unit of the same source).
#define ATTN_BWD_HEAD_DIM 128
#define ATTN_BWD_VALUE_DIM 64
#include "bwd_tcgen05.cu"
