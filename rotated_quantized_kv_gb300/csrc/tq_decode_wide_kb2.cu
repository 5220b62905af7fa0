// tq_decode_wide_kb2.cu -- split-K decode kernels for packed segments with
// 2-bit keys at head_dim 256 and 512 (every value width).
#include "tq_decode_packed.cuh"

TQ_INSTANTIATE_WIDE_KB(2)
