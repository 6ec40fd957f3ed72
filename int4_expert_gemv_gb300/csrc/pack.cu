// pack.cu -- builds packed records / expert blobs from logical tensors, and the
// decode test hook.
//
// Logical input of one matrix: codes q uint32 [rows][cols*bits/32] (element j
// of a word at bits [bits*j, bits*j+bits)), fp16 scales s and biases b
// [rows][cols/64].  Output record of a row: the same code words, then the
// {s, b} pairs of its groups interleaved, then zero padding to 16 bytes.
#include "internal.h"

namespace moe {

// One warp per (row, matrix): grid (ceil(rows / 8), nmat), block 256.
// Row i of matrix m goes to record first_record + i*record_step of
// dst + m*dst_mat_stride.
__global__ void __launch_bounds__(256) pack_rows_kernel(
    const uint32_t *q, const uint16_t *s, const uint16_t *b, int rows, int cols, int bits,
    size_t src_q_stride, size_t src_sb_stride, uint8_t *dst, size_t dst_mat_stride,
    size_t first_record, size_t record_step, size_t rec) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * (blockDim.x >> 5) + warp;
    const int m = blockIdx.y;
    if (row >= rows) return;
    const int words = cols * bits / 32, groups = cols / kGroup;
    const uint32_t *qr = q + m * src_q_stride + (size_t)row * words;
    const uint16_t *sr = s + m * src_sb_stride + (size_t)row * groups;
    const uint16_t *br = b + m * src_sb_stride + (size_t)row * groups;
    uint8_t *out = dst + m * dst_mat_stride + (first_record + (size_t)row * record_step) * rec;
    uint32_t *ow = reinterpret_cast<uint32_t *>(out);
    for (int i = lane; i < words; i += 32) ow[i] = qr[i];
    for (int g = lane; g < groups; g += 32)
        ow[words + g] = (uint32_t)sr[g] | ((uint32_t)br[g] << 16);
    for (int i = words + groups + lane; i < (int)(rec / 4); i += 32) ow[i] = 0u;
}

int launch_pack_rows(const uint32_t *q, const uint16_t *s, const uint16_t *b, int rows,
                     int cols, int bits, int nmat, size_t src_q_stride, size_t src_sb_stride,
                     uint8_t *dst, size_t dst_mat_stride, size_t first_record,
                     size_t record_step, cudaStream_t st) {
    dim3 grid((rows + 7) / 8, nmat);
    pack_rows_kernel<<<grid, 256, 0, st>>>(q, s, b, rows, cols, bits, src_q_stride,
                                           src_sb_stride, dst, dst_mat_stride, first_record,
                                           record_step, record_bytes(cols, bits));
    return check_launch("pack_rows_kernel");
}

// out[r][c] = fmaf(code, scale, bias) for record first_record + r*record_step.
__global__ void debug_dequant_kernel(const uint8_t *sec, size_t rec, size_t first_record,
                                     size_t record_step, int rows, int cols, int bits,
                                     float *out) {
    const size_t n = (size_t)rows * cols;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x) {
        const int r = (int)(i / cols), c = (int)(i % cols);
        const uint8_t *rp = sec + (first_record + (size_t)r * record_step) * rec;
        const int per = 32 / bits;
        const uint32_t w = reinterpret_cast<const uint32_t *>(rp)[c / per];
        const uint32_t code = (w >> (bits * (c % per))) & ((1u << bits) - 1u);
        const uint32_t sbw =
            reinterpret_cast<const uint32_t *>(rp + code_bytes(cols, bits))[c / kGroup];
        const float2 sb = sb_f(sbw);
        out[i] = fmaf(code_f(code), sb.x, sb.y);
    }
}

int launch_debug_dequant(const uint8_t *sec, size_t rec, size_t first_record,
                         size_t record_step, int rows, int cols, int bits, float *out,
                         cudaStream_t st) {
    const size_t n = (size_t)rows * cols;
    const int blocks = (int)((n + 255) / 256 < 65535 ? (n + 255) / 256 : 65535);
    debug_dequant_kernel<<<blocks, 256, 0, st>>>(sec, rec, first_record, record_step, rows,
                                                 cols, bits, out);
    return check_launch("debug_dequant_kernel");
}

}  // namespace moe
