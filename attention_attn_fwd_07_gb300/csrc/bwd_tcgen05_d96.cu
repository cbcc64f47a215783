// bwd_tcgen05_d96.cu -- the attention backward kernels of bwd_tcgen05.cu
// built for head dim 96, key and value (a translation unit of the same
// source): Q/K/V/dO tiles of two swizzle atoms, the second half zero-filled
// by the tensor maps, six MMA K steps for S and dP, N = 96 for dK, dV, dQ.
#define ATTN_BWD_HEAD_DIM 96
#include "bwd_tcgen05.cu"
