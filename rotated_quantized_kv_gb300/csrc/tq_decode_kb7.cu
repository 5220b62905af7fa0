// tq_decode_kb7.cu -- split-K decode kernels for packed segments with
// 7-bit keys (every value width, with and without the QJL term).
#include "tq_decode_packed.cuh"

TQ_INSTANTIATE_PACKED_KB(7)
