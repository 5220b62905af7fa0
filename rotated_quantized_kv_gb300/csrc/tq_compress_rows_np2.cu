// tq_compress_rows_np2.cu -- the one-thread-per-slice compressor at head_dim 64
// (two tokens per thread, tq_compress_rows.cuh).
#include "tq_compress_rows.cuh"

namespace tqk {

cudaError_t launch_compress_rows_np2(const RowsParams &p, int bits, bool values, cudaStream_t s) {
    return rows_dispatch<1, 2>(p, bits, values, s);
}

}  // namespace tqk
