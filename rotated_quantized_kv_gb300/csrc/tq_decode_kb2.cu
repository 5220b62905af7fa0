// tq_decode_kb2.cu -- split-K decode kernels for packed segments with
// 2-bit keys (every value width, with and without the QJL term).
#include "tq_decode_packed.cuh"

TQ_INSTANTIATE_PACKED_KB(2)
