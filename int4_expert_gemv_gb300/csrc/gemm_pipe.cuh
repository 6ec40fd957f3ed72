// gemm_pipe.cuh -- persistent, warp-specialised tensor-core GEMM of packed
// group-64 affine records (4- or 2-bit codes) against bf16 activation rows,
// for several tokens at once.  Shared by the batched expert FFN (gate/up,
// down) and the batched prerouter head (fc1 and l on x).
//
// A job describes the work as items: kRB consecutive records against up to
// kTok consecutive activation rows.  One CTA per SM runs items b, b + grid,
// ...; their 256-column chunks stream through a kStages-deep ring in shared
// memory.  One producer warp fills the ring with TMA tensor copies (the
// codes and the {scale, bias} words of the item's records from 3-D maps over
// the packed weights, the activation rows and their per-group sums in boxes
// of 8 rows), completing on a per-stage "full" mbarrier; sixteen consumer
// warps -- two per 16 records, each taking half of a chunk's columns -- run
// the MMAs and release the stage on its "empty" mbarrier.  Item boundaries
// do not drain the ring.
//
// The MMA (m16n8k16, bf16 in, fp32 accumulate) takes the codes themselves:
// offset into one binade a code is exact in bf16 and formed by an OR -- a
// 4-bit q as 16 + q (bits 0x4180 | q << 3), a 2-bit q as 4 + q (bits
// 0x4080 | q << 5).  Per 64-column group (scale s, bias b, offset c) the
// affine terms are applied in fp32:
//   sum_k (q_k s + b) x_k = s * sum (c + q) x + (b - c s) * sum x,
// so dequantised weights are never rounded.  An item issues the MMAs (and
// the activation copies) of its real tokens only, in n-tiles of 8: with one
// token it costs its weight bytes and little more (a weight-streaming GEMV),
// with many it is a GEMM.
//
// Every wait is bounded: on expiry the waiting warp records MOE_ETIMEOUT in
// the job's error word and runs on without waiting (its results are then
// garbage), and the producer finally waits, again bounded, for the copies
// it issued, so no CTA exits with a copy in flight and no launch hangs.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "common.cuh"

namespace moe {
namespace pipe {

constexpr int kTok = 64;          // activation rows per item (up to 8 n-tiles of 8)
constexpr int kKc = 256;          // columns per chunk (4 groups of 64)
constexpr int kGpc = kKc / kGroup;
constexpr int kRB = 128;          // records per item (8 row warps x m16)
constexpr int kRowWarps = kRB / 16;
constexpr int kConsumers = 2 * kRowWarps;   // two warps per 16 records, each half the columns
constexpr int kThr = (kConsumers + 1) * 32;
constexpr int kStages = 4;
constexpr int kRowBox = 8;        // activation rows per TMA box

// Stage layout in bytes; every part starts on a 128-byte boundary.
constexpr int kSbOff = kRB * kKc / 2;          // codes: kRB x (kKc * BITS / 8), dense
constexpr int kXOff = kSbOff + kRB * 16;       // {s, b}: kRB x 4 groups x 4 bytes
constexpr int kXRow = kKc * 2;                 // one activation row of the chunk (bf16)
constexpr int kXsOff = kXOff + kTok * kXRow;   // activations: kTok x kXRow
constexpr int kEntOff = kXsOff + kTok * 16;    // group sums: kTok x 4 floats
constexpr int kStageB = ((kEntOff + kTok * 4) + 1023) / 1024 * 1024;
constexpr int kOutLd = kTok + 1;               // epilogue staging row (floats)
static_assert(kRB * kOutLd * 4 <= kEntOff, "the epilogue staging would overwrite the entries");
static_assert(kXOff % 1024 == 0 && kTok * kXRow == 4 * kTok * 128,
              "activation slabs of 64 columns on 1 KB swizzle atoms");

constexpr uint64_t kDefaultWaitNs = 1000000000ull;   // a wait's bound unless set

// Bounds of the engine's device-side waits, process-wide (host side):
// timeout_ns (0 = kDefaultWaitNs) and a test hook -- stall != 0 makes
// consumer warp 0 of CTA 0 wait for bytes no copy sends, so that wait runs
// out and the launch takes its expiry path.
struct WaitCfg {
    unsigned long long timeout_ns;
    int stall;
};
inline WaitCfg &wait_cfg() {
    static WaitCfg w{0, 0};
    return w;
}

// Offset c of the bf16 code values (c + q).
template <int BITS> struct CodeOff;
template <> struct CodeOff<4> { static constexpr float c = 16.0f; };
template <> struct CodeOff<2> { static constexpr float c = 4.0f; };

// An item: group g, row block rb, tokens t0 .. t0 + nt - 1 of the group.
struct Item {
    int g, rb, t0, nt;
};

// The tensor maps of a job: weight records of two sources (map 0: the
// indexed blobs, map 1: a single blob), codes and {s, b} boxes of each; the
// activation rows; their per-group sums.
struct Maps {
    CUtensorMap codes[2], sb[2], act, gsum;
    // for the tcgen05 engine (gemm_umma.cuh): the codes of a chunk (4-bit:
    // one 128-byte box per record, 128-byte swizzle; 2-bit: one 16-byte box
    // per record and group), activations in 64-column boxes with the 128-byte
    // swizzle of the tensor cores' K-major operand layout and their group
    // sums, each in boxes of 8, 16, 32 or 64 rows
    CUtensorMap gcodes[2], act128[4], gsum4[4];
    // the register engine's activations in boxes of 8, 16, 32 or 64 rows
    CUtensorMap act4[4];
};

// ---------------------------------------------------------------- host
inline PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

inline int encode_map(CUtensorMap *m, CUtensorMapDataType dt, int rank, const void *base,
                      const cuuint64_t *dims, const cuuint64_t *strides, const cuuint32_t *box,
                      CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE) {
    const PFN_cuTensorMapEncodeTiled_v12000 fn = tmap_encoder();
    if (fn == nullptr) return MOE_ECUDA;
    const cuuint32_t es[5] = {1, 1, 1, 1, 1};
    const CUresult r = fn(m, dt, (cuuint32_t)rank, const_cast<void *>(base), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MOE_OK : MOE_ECUDA;
}

// Records of `nblobs` blobs: record r of blob z at base + z * blob_stride +
// r * rec; nrows records per blob.
inline int weight_maps(Maps &m, int which, const void *base, size_t rec, int nrows, int nblobs,
                       size_t blob_stride, int bits) {
    if (nblobs == 1) blob_stride = rec * (size_t)nrows;
    const cuuint64_t dims[3] = {rec, (cuuint64_t)nrows, (cuuint64_t)nblobs};
    const cuuint64_t strides[2] = {rec, blob_stride};
    const cuuint32_t bc[3] = {(cuuint32_t)(kKc * bits / 8), kRB, 1};
    const cuuint32_t bs[3] = {16, kRB, 1};
    if (int rc = encode_map(&m.codes[which], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, bc))
        return rc;
    if (bits == 4) {
        if (int rc = encode_map(&m.gcodes[which], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, bc,
                                CU_TENSOR_MAP_SWIZZLE_128B))
            return rc;
    } else {
        const cuuint32_t bg[3] = {(cuuint32_t)(kGroup * bits / 8), kRB, 1};
        if (int rc = encode_map(&m.gcodes[which], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, bg))
            return rc;
    }
    return encode_map(&m.sb[which], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, bs);
}

// Row stride (floats) of a per-group sum array of `cols` columns: padded to
// 16 bytes, as a tensor map requires.
__host__ __device__ inline int gsum_ld(int cols) { return (cols / kGroup + 3) / 4 * 4; }

// Activation rows (bf16, rows x cols) and their per-group sums.
inline int act_maps(Maps &m, const void *act, const float *gsum, int rows, int cols) {
    const cuuint64_t da[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t sa[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t ba[2] = {kKc, kRowBox};
    if (int rc = encode_map(&m.act, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, act, da, sa, ba)) return rc;
    const cuuint64_t dg[2] = {(cuuint64_t)(cols / kGroup), (cuuint64_t)rows};
    const cuuint64_t sg[1] = {(cuuint64_t)gsum_ld(cols) * 4};
    for (int i = 0; i < 4; i++) {                  // boxes of 8 << i rows
        const cuuint32_t bai[2] = {kKc, (cuuint32_t)(kRowBox << i)};
        if (int rc = encode_map(&m.act4[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, act, da, sa, bai)) return rc;
        const cuuint32_t b128[2] = {kGroup, (cuuint32_t)(kRowBox << i)};
        if (int rc = encode_map(&m.act128[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, act, da, sa, b128,
                                CU_TENSOR_MAP_SWIZZLE_128B))
            return rc;
        const cuuint32_t bgi[2] = {kGpc, (cuuint32_t)(kRowBox << i)};
        if (int rc = encode_map(&m.gsum4[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, gsum, dg, sg, bgi))
            return rc;
    }
    const cuuint32_t bg[2] = {kGpc, kRowBox};
    return encode_map(&m.gsum, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, gsum, dg, sg, bg);
}

// ---------------------------------------------------------------- device
__device__ __forceinline__ uint32_t saddr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(bar)),
                 "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; "
        "selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(saddr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait of a whole warp for the phase of `bar` with `parity`: lane 0
// polls (for at most timeout_ns), the outcome is shared, then every lane
// observes the completed phase itself (its acquire of the stage's data).
// Returns false on expiry.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, uint64_t timeout_ns) {
    uint32_t ok = 0;
    if ((threadIdx.x & 31) == 0) {
        ok = mbar_try_wait(bar, parity);
        const uint64_t t0 = ok ? 0 : globaltimer_ns();
        for (uint32_t i = 1; !ok; i++) {
            ok = mbar_try_wait(bar, parity);
            if (!ok && (i & 15) == 0 && globaltimer_ns() - t0 > timeout_ns) break;
        }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) mbar_try_wait(bar, parity);
    return ok != 0;
}

__device__ __forceinline__ void consumers_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory");
}

__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void tma_3d(void *dst, const CUtensorMap *m, int x, int y, int z,
                                       uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;"
        ::"r"(saddr(dst)), "l"(m), "r"(x), "r"(y), "r"(z), "r"(saddr(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_2d(void *dst, const CUtensorMap *m, int x, int y,
                                       uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        ::"r"(saddr(dst)), "l"(m), "r"(x), "r"(y), "r"(saddr(bar))
        : "memory");
}

// (not volatile: a pure function of its operands, so the compiler may
// interleave the independent MMAs of different n-tiles)
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// bf16 pair for byte b of two pre-shifted code words lo, hi: byte b of lo
// into the low half, byte b of hi into the high half, masked, with the
// offset's exponent bits or'ed in.
__device__ __forceinline__ uint32_t pair_from(uint32_t lo, uint32_t hi, int b, uint32_t mask,
                                              uint32_t one) {
    const uint32_t t = __byte_perm(lo, hi, (uint32_t)(b | (b << 4) | ((4 + b) << 8) | ((4 + b) << 12)));
    return (t & mask) | one;
}

// A fragments of one 64-column group for the warp's records r0 and r0 + 8:
// a[ks][0..3] for the 4 MMA k-steps.  Within a group the MMA's k index maps
// to column 16 j + 4 ks + 2 (k / 8) + k % 2 (j = k % 8 / 2, the lane's
// position in its quad), the same map for A and B, so that a lane's codes
// are contiguous (4-bit: 8 bytes per record; 2-bit: 4 bytes) and so are its
// activations (16 bf16 per token).
template <int BITS>
__device__ __forceinline__ void a_frags(const uint8_t *codes, int r0, int gi, int j,
                                        uint32_t (&a)[4][4]) {
    constexpr int CB = kKc * BITS / 8;
    if (BITS == 4) {
#pragma unroll
        for (int h = 0; h < 2; h++) {          // record r0 (h = 0), r0 + 8 (h = 1)
            // records of 128 bytes with the 128-byte swizzle: 16-byte piece c
            // of record r at 16 (c ^ r % 8)
            const int r = r0 + 8 * h, o = gi * 32 + j * 8;
            const uint2 w = *reinterpret_cast<const uint2 *>(codes + r * CB + ((((o >> 4) ^ (r & 7)) << 4) | (o & 15)));
#pragma unroll
            for (int half = 0; half < 2; half++) {   // columns 16j + 0..7, 16j + 8..15
                const uint32_t v = half ? w.y : w.x;
                const uint32_t ev = (v << 3) & 0x78787878u, od = (v >> 1) & 0x78787878u;
#pragma unroll
                for (int kk = 0; kk < 2; kk++) {
                    const int ks = 2 * half + kk;
                    a[ks][h] = pair_from(ev, od, 2 * kk, 0x00780078u, 0x41804180u);
                    a[ks][2 + h] = pair_from(ev, od, 2 * kk + 1, 0x00780078u, 0x41804180u);
                }
            }
        }
    } else {
#pragma unroll
        for (int h = 0; h < 2; h++) {
            const uint32_t v = *reinterpret_cast<const uint32_t *>(codes + (r0 + 8 * h) * CB + gi * 16 + j * 4);
            const uint32_t c0 = (v << 5) & 0x60606060u, c1 = (v << 3) & 0x60606060u;
            const uint32_t c2 = (v << 1) & 0x60606060u, c3 = (v >> 1) & 0x60606060u;
#pragma unroll
            for (int ks = 0; ks < 4; ks++) {
                a[ks][h] = pair_from(c0, c1, ks, 0x00600060u, 0x40804080u);
                a[ks][2 + h] = pair_from(c2, c3, ks, 0x00600060u, 0x40804080u);
            }
        }
    }
}

// The MMAs of groups g0 .. g1 - 1 (64 columns each) of one staged chunk
// for the warp's 16 records rw*16 .., nnt n-tiles of 8 tokens; the affine
// terms of each group are folded into total.  total[nti][q] is the warp's
// fragment: record rw*16 + lane/4 (+8 for q >= 2), token
// nti*8 + 2*(lane%4) + (q & 1).
template <int BITS>
__device__ __forceinline__ void mma_chunk(const uint8_t *stage, int rw, int g0, int g1, int nnt,
                                          float (&total)[8][4]) {
    const int lane = threadIdx.x & 31;
    const int r0 = rw * 16 + (lane >> 2), j = lane & 3, gq = lane >> 2;
    const uint32_t *sb = reinterpret_cast<const uint32_t *>(stage + kSbOff);
    const __nv_bfloat16 *x = reinterpret_cast<const __nv_bfloat16 *>(stage + kXOff);
    const float *xs = reinterpret_cast<const float *>(stage + kXsOff);
#pragma unroll 1
    for (int gi = g0; gi < g1; gi++) {
        uint32_t a[4][4];
        a_frags<BITS>(stage, r0, gi, j, a);
        const float2 sb0 = sb_f(sb[r0 * kGpc + gi]), sb1 = sb_f(sb[(r0 + 8) * kGpc + gi]);
        constexpr float off = CodeOff<BITS>::c;
        const float c0 = fmaf(-off, sb0.x, sb0.y), c1 = fmaf(-off, sb1.x, sb1.y);
#pragma unroll
        for (int nti = 0; nti < 8; nti++) {
            if (nti < nnt) {
                // group gi's activation rows: 128 bytes each, 128-byte swizzle
                // (16-byte piece c of row t at 16 (c ^ t % 8)); this lane's 16
                // values are pieces 2j and 2j + 1
                const int t = nti * 8 + gq;
                const uint8_t *xr = reinterpret_cast<const uint8_t *>(x) + gi * (kTok * 128) + t * 128;
                const uint4 xa = *reinterpret_cast<const uint4 *>(xr + (((2 * j) ^ (t & 7)) << 4));
                const uint4 xb = *reinterpret_cast<const uint4 *>(xr + (((2 * j + 1) ^ (t & 7)) << 4));
                float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                mma_bf16(acc, a[0], xa.x, xa.y);
                mma_bf16(acc, a[1], xa.z, xa.w);
                mma_bf16(acc, a[2], xb.x, xb.y);
                mma_bf16(acc, a[3], xb.z, xb.w);
                // affine terms of the group: s * acc + (b - c s) * sum x
                const float x0 = xs[(nti * 8 + 2 * j) * kGpc + gi];
                const float x1 = xs[(nti * 8 + 2 * j + 1) * kGpc + gi];
                total[nti][0] = fmaf(sb0.x, acc[0], fmaf(c0, x0, total[nti][0]));
                total[nti][1] = fmaf(sb0.x, acc[1], fmaf(c0, x1, total[nti][1]));
                total[nti][2] = fmaf(sb1.x, acc[2], fmaf(c1, x0, total[nti][2]));
                total[nti][3] = fmaf(sb1.x, acc[3], fmaf(c1, x1, total[nti][3]));
            }
        }
    }
}

// The persistent kernel.  Job supplies (device, const):
//   maps (Maps), cols, err (int32_t *, the error word),
//   init(sm): copies what item() reads into the shared scratch sm,
//   n_items(sm), item(sm, i),
//   weights(it, map, row, blob): the tensor-map coordinates of its records,
//   row0(sm, it): its first activation row (the rest follow),
//   meta(sm, it): nt words for the epilogue (or null),
//   epilogue(sm, it, out, ent, tid, nthr): out[r * kOutLd + t] = record r's
//     dot with token t; tid in [0, nthr) of the threads that run it.
// Dynamic shared memory: alignment slack, kStages stages, 2 kStages
// mbarriers, the scratch.
template <int BITS, class Job>
__global__ void __launch_bounds__(kThr, 1) pipe_gemm_kernel(const __grid_constant__ Job job,
                                                            const uint64_t timeout_ns, const int stall) {
    extern __shared__ __align__(1024) uint8_t smdyn[];
    // stages on a 1024-byte boundary (TMA destinations), whatever the base
    uint8_t *smraw = smdyn + ((1024u - (saddr(smdyn) & 1023u)) & 1023u);
    uint64_t *full = reinterpret_cast<uint64_t *>(smraw + kStages * kStageB);
    uint64_t *empty = full + kStages;
    uint64_t *stall_bar = empty + kStages;          // the test hook's wait
    int32_t *sm = reinterpret_cast<int32_t *>(stall_bar + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; s++) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, kConsumers);
        }
        mbar_init(stall_bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    job.init(sm);
    __syncthreads();
    const int n_items = job.n_items(sm);
    const int b = blockIdx.x, nb = gridDim.x;
    const int mine = n_items > b ? (n_items - 1 - b) / nb + 1 : 0;
    const int nch = (job.cols + kKc - 1) / kKc;
    const int nq = mine * nch;
    constexpr uint32_t kCodeBytes = kRB * kKc * BITS / 8;

    if (warp == kConsumers) {
        // ------------------------------------------------ producer
        const uint64_t policy = evict_first_policy();
        const int cbytes = job.cols * BITS / 8;
        int li = 0, lc = 0;
        Item it = nq > 0 ? job.item(sm, b) : Item{};
        int q = 0;
        for (; q < nq; q++) {
            const int s = q % kStages;
            uint8_t *stage = smraw + s * kStageB;
            if (q >= kStages && !warp_wait(empty + s, ((q / kStages) - 1) & 1, timeout_ns)) {
                if (lane == 0) atomicExch(job.err, MOE_ETIMEOUT);
                break;
            }
            if (lc == nch - 1) {            // the item's last chunk carries its entries
                const int32_t *m = job.meta(sm, it);
                int32_t *ent = reinterpret_cast<int32_t *>(stage + kEntOff);
                if (m != nullptr)
                    for (int t = lane; t < it.nt; t += 32) ent[t] = m[t];
            }
            // the chunk's copies, each from a lane of its own (one lane issues a
            // copy only every ~200 ns): the codes (4-bit: 128-byte records with
            // the 128-byte swizzle), {s, b}, per group the activation rows (in
            // one box of 8, 16, 32 or 64 rows, 128-byte swizzle), their group
            // sums
            const int ng = min(kKc, job.cols - lc * kKc) / kGroup;
            const int bk = it.nt <= 8 ? 0 : it.nt <= 16 ? 1 : it.nt <= 32 ? 2 : 3;
            const int rows = kRowBox << bk;
            if (lane == 0) mbar_expect_tx(full + s, kCodeBytes + kRB * 16 + ng * rows * 128 + rows * 16);
            __syncwarp();
            int map, row, blob;
            job.weights(it, map, row, blob);
            const int r0 = job.row0(sm, it);
            if (lane == 0)
                tma_3d(stage, BITS == 4 ? &job.maps.gcodes[map] : &job.maps.codes[map], lc * kKc * BITS / 8,
                       row, blob, full + s, policy);
            else if (lane == 1)
                tma_3d(stage + kSbOff, &job.maps.sb[map], cbytes + 16 * lc, row, blob, full + s, policy);
            else if (lane < 2 + ng)
                tma_2d(stage + kXOff + (lane - 2) * (kTok * 128), &job.maps.act128[bk],
                       lc * kKc + (lane - 2) * kGroup, r0, full + s);
            else if (lane == 2 + ng)
                tma_2d(stage + kXsOff, &job.maps.gsum4[bk], lc * kGpc, r0, full + s);
            if (++lc == nch) {
                lc = 0;
                if (++li < mine) it = job.item(sm, b + li * nb);
            }
        }
        // the copies of the last fill of each stage land before the CTA exits
        for (int s = 0; s < kStages && s < q; s++) {
            const int last = q - 1 - ((q - 1 - s) % kStages);     // last chunk issued on s
            if (!warp_wait(full + s, (last / kStages) & 1, timeout_ns) && lane == 0)
                atomicExch(job.err, MOE_ETIMEOUT);
        }
        return;
    }

    // ---------------------------------------------------- consumers
    // warp w: records (w % 8) * 16 .., column groups 2 (w / 8), 2 (w / 8) + 1
    const int tid = threadIdx.x, rw = warp % kRowWarps, kh = warp / kRowWarps;
    bool dead = false;
    if (stall && blockIdx.x == 0 && warp == 0) {
        // test hook: 16 bytes that no copy sends; the wait runs out and this
        // warp goes on as a warp whose stage never arrived
        if (lane == 0) mbar_expect_tx(stall_bar, 16);
        __syncwarp();
        if (!warp_wait(stall_bar, 0, timeout_ns)) {
            dead = true;
            if (lane == 0) atomicExch(job.err, MOE_ETIMEOUT);
        }
    }
    float total[8][4];
#pragma unroll
    for (int u = 0; u < 8; u++)
#pragma unroll
        for (int v = 0; v < 4; v++) total[u][v] = 0.0f;
    int ci = 0, cc = 0;
    Item it = nq > 0 ? job.item(sm, b) : Item{};
#pragma unroll 1
    for (int q = 0; q < nq; q++) {
        const int s = q % kStages;
        uint8_t *stage = smraw + s * kStageB;
        if (!dead && !warp_wait(full + s, (q / kStages) & 1, timeout_ns)) {
            dead = true;
            if (lane == 0) atomicExch(job.err, MOE_ETIMEOUT);
        }
        const int gc = min(kKc, job.cols - cc * kKc) / kGroup;
        mma_chunk<BITS>(stage, rw, min(gc, 2 * kh), min(gc, 2 * kh + 2), (it.nt + 7) >> 3, total);
        if (++cc == nch) {
            // stage the item's results in the stage (all its reads are done):
            // the first column half stores, the second adds
            float *out = reinterpret_cast<float *>(stage);
            const int gq = lane >> 2, j = lane & 3, nnt = (it.nt + 7) >> 3;
#pragma unroll
            for (int h = 0; h < 2; h++) {
                consumers_sync();
                if (kh == h) {
#pragma unroll
                    for (int nti = 0; nti < 8; nti++)
                        if (nti < nnt)
#pragma unroll
                            for (int u = 0; u < 4; u++) {
                                float &o = out[(rw * 16 + gq + 8 * (u >> 1)) * kOutLd + nti * 8 + 2 * j + (u & 1)];
                                o = h ? o + total[nti][u] : total[nti][u];
                            }
                }
            }
            consumers_sync();
            job.epilogue(sm, it, out, reinterpret_cast<const int32_t *>(stage + kEntOff), tid,
                         kConsumers * 32);
#pragma unroll
            for (int u = 0; u < 8; u++)
#pragma unroll
                for (int v = 0; v < 4; v++) total[u][v] = 0.0f;
            cc = 0;
            if (++ci < mine) it = job.item(sm, b + ci * nb);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty + s);
    }
}

// Launches the persistent kernel on every SM.  scratch_bytes: the job's
// shared-memory scratch.
template <int BITS, class Job>
inline int launch_pipe_gemm(const Job &job, size_t scratch_bytes, int sms, cudaStream_t st,
                            const char *name) {
    const size_t smem = 1024 + (size_t)kStages * kStageB + (2 * kStages + 1) * sizeof(uint64_t) +
                        scratch_bytes;
    cudaFuncSetAttribute(pipe_gemm_kernel<BITS, Job>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
    const WaitCfg w = wait_cfg();
    pipe_gemm_kernel<BITS, Job><<<sms, kThr, smem, st>>>(job, w.timeout_ns ? w.timeout_ns : kDefaultWaitNs,
                                                          w.stall);
    return check_launch(name);
}

// sums[r * ld + g] = sum of v[r][64 g .. 64 g + 63] (bf16 values, fp32 sum
// in a fixed order), rows r < rows, ld = gsum_ld(cols).  One warp per
// (row, group).
static __global__ void __launch_bounds__(256) group_sums_kernel(const __nv_bfloat16 *v, int rows,
                                                                int cols, float *sums) {
    const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    const int ng = cols / kGroup;
    if (w >= rows * ng) return;
    const int r = w / ng, g = w - (w / ng) * ng;
    const __nv_bfloat162 p = reinterpret_cast<const __nv_bfloat162 *>(v + (size_t)r * cols + g * kGroup)[lane];
    float a = __bfloat162float(p.x) + __bfloat162float(p.y);
    a = warp_sum(a, 32);
    if (lane == 0) sums[(size_t)r * gsum_ld(cols) + g] = a;
}

inline int launch_group_sums(const __nv_bfloat16 *v, int rows, int cols, float *sums,
                             cudaStream_t st) {
    const int warps = rows * (cols / kGroup);
    group_sums_kernel<<<(warps + 7) / 8, 256, 0, st>>>(v, rows, cols, sums);
    return check_launch("group_sums_kernel");
}

}  // namespace pipe
}  // namespace moe
