// bwd_tcgen05_d64.cu -- the attention backward kernels of bwd_tcgen05.cu
// built for head dim 64 (a second translation unit of the same source).
#define ATTN_BWD_HEAD_DIM 64
#include "bwd_tcgen05.cu"
