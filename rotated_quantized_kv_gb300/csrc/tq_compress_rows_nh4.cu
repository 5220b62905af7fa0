// tq_compress_rows_nh4.cu -- the one-thread-per-slice compressor at head_dim
// 512 (4 slices per vector, tq_compress_rows.cuh).
#include "tq_compress_rows.cuh"

namespace tqk {

cudaError_t launch_compress_rows_nh4(const RowsParams &p, int bits, bool values, cudaStream_t s) {
    return rows_dispatch<4>(p, bits, values, s);
}

}  // namespace tqk
