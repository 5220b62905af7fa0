// tq_compress_rows_nh2.cu -- the one-thread-per-slice compressor at head_dim
// 256 (2 slices per vector, tq_compress_rows.cuh).
#include "tq_compress_rows.cuh"

namespace tqk {

cudaError_t launch_compress_rows_nh2(const RowsParams &p, int bits, bool values, cudaStream_t s) {
    return rows_dispatch<2>(p, bits, values, s);
}

}  // namespace tqk
