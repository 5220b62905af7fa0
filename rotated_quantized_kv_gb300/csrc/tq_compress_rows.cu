// tq_compress_rows.cu -- the one-thread-per-slice compressor at head_dim 128
// and the dispatch over the slice counts (tq_compress_rows.cuh).
#include "tq_compress_rows.cuh"

namespace tqk {

cudaError_t launch_compress_rows(const RowsParams &p, int bits, bool values, cudaStream_t s) {
    if (p.np == 2) return launch_compress_rows_np2(p, bits, values, s);
    switch (p.nh) {
        case 1: return rows_dispatch<1>(p, bits, values, s);
        case 2: return launch_compress_rows_nh2(p, bits, values, s);
        case 4: return launch_compress_rows_nh4(p, bits, values, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace tqk
