// gemm_umma.cuh -- the batched engine on the 5th-generation tensor cores:
// tcgen05.mma with the accumulator in tensor memory (TMEM).
//
// The same jobs, items and TMA streams as gemm_pipe.cuh (kRB = 128 records
// against up to kTok = 64 activation rows, 256-column chunks through a ring
// of stages), with the math moved off the registers:
//   * converter warps turn each 64-column group of packed codes into a bf16
//     A tile in shared memory -- the code offset into one binade, c + q,
//     exact in bf16 and formed by an OR -- in the canonical K-major layout
//     with the 128-byte swizzle;
//   * one thread issues tcgen05.mma (kind::f16, bf16 x bf16 -> fp32, M = 128,
//     N = the item's tokens rounded up to 16, K = 16 per instruction, 4 per
//     group) from that tile and the group's activation tile (loaded by TMA in
//     the same swizzled layout) into one of two TMEM accumulators;
//   * epilogue warps read the group's accumulator (tcgen05.ld), apply the
//     group's affine terms exactly as the register engine does,
//       sum_k (q_k s + b) x_k = s * sum (c + q) x + (b - c s) * sum x,
//     and keep each record's running total in registers (one record per
//     thread, the thread's TMEM lane).
// kSlots A tiles and accumulators rotate, so the conversion of later groups
// and their MMAs run while group g's accumulator is read back and folded.  A per-group
// accumulator is what keeps the dequantised weights unrounded: the scale of a
// group multiplies its exact bf16 partial sum in fp32.
//
// Warp roles (320 threads): warps 0-3 epilogue (warp w owns TMEM lanes and
// records 32w .. 32w + 31), warps 4-7 converters (thread = record), warp 8
// MMA issue and TMEM allocation, warp 9 the TMA producer.  Every wait is
// bounded; the first one to expire records MOE_ETIMEOUT in the job's error
// word and raises an abort flag in shared memory, after which no role waits
// or issues MMAs any more, the producer waits (bounded) for the copies it
// issued, and the CTA frees its TMEM and exits.
#pragma once

#include "gemm_pipe.cuh"

namespace moe {
namespace umma {

using pipe::Item;
using pipe::kGpc;
using pipe::kKc;
using pipe::kRB;
using pipe::kRowBox;
using pipe::kTok;

constexpr int kEpiWarps = 4;
constexpr int kCvtWarps = 4;
constexpr int kMmaWarp = kEpiWarps + kCvtWarps;
constexpr int kProdWarp = kMmaWarp + 1;
constexpr int kThreads = (kProdWarp + 1) * 32;
constexpr int kStages = 3;
constexpr int kSlots = 4;                 // A tiles and TMEM accumulators in flight
constexpr int kPer = 2;                   // groups per handoff (a bank of slots)
constexpr int kBanks = kSlots / kPer;
constexpr int kAccCols = 64;              // fp32 columns of one accumulator (kTok tokens)
constexpr int kTmemCols = kSlots * kAccCols;

// Stage layout (bytes).  Codes: 4-bit, kRB records x 128 bytes (the chunk's
// 4 groups) with the 128-byte swizzle; 2-bit, per group kRB records x 16
// bytes, unswizzled.  {s, b}: kRB x 16 bytes.
// Activations: per group, kTok rows x 128 bytes (64 bf16), 128-byte swizzle,
// one 1 KB atom per 8 rows.  Then per-group sums (kTok x 16 bytes) and the
// item's entry words.
constexpr int kCodeGroup = kRB * 32;
constexpr int kSbOff = 4 * kCodeGroup;
constexpr int kXOff = kSbOff + kRB * 16;
constexpr int kXGroup = kTok * 128;
constexpr int kXsOff = kXOff + 4 * kXGroup;
constexpr int kEntOff = kXsOff + kTok * 16;
constexpr int kStageB = (kEntOff + kTok * 4 + 1023) / 1024 * 1024;
constexpr int kOutLd = kTok + 1;
static_assert(kOutLd == pipe::kOutLd, "the jobs' epilogues read the staging with pipe::kOutLd");
constexpr int kSlotB = kRB * 128;          // one A tile: 128 records x 64 bf16, swizzled
static_assert(kXOff % 1024 == 0 && kXGroup % 1024 == 0, "swizzled tiles sit on 1 KB atoms");
static_assert(kTmemCols <= 512 && (kTmemCols & (kTmemCols - 1)) == 0, "a TMEM allocation");
static_assert(kSlots == kPer * kBanks && kBanks >= 2, "banks of slots, double-buffered");
static_assert(kRB * kOutLd * 4 <= kEntOff - kXOff,
              "the item's results are staged over its last chunk's activations and sums");
constexpr int kBars = 2 * kStages + 4 * kBanks + 1;
constexpr size_t kFixedSmem = 1024 + (size_t)kStages * kStageB + (size_t)kSlots * kSlotB +
                              kBars * 8 + 16;

// ---------------------------------------------------------------- device
using pipe::globaltimer_ns;
using pipe::mbar_arrive;
using pipe::mbar_expect_tx;
using pipe::mbar_init;
using pipe::mbar_try_wait;
using pipe::pair_from;
using pipe::saddr;
using pipe::tma_2d;
using pipe::tma_3d;

// Shared-memory matrix descriptor of a K-major tile in the canonical
// 128-byte-swizzle layout: rows of 128 bytes, 8-row atoms 1024 bytes apart
// (stride byte offset), start address encoded >> 4, descriptor version 1,
// swizzle mode 2 (128 bytes).  The leading byte offset is unused by this
// layout (K per instruction stays inside one atom) and set to 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t smem_addr) {
    return (uint64_t)((smem_addr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) |
           ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator (bits 4-5 = 1), A and
// B bf16 (bits 7-9, 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 in
// bits 17-22, M >> 4 in bits 24-28 (M = 128).
__device__ __forceinline__ uint32_t idesc_bf16_m128(int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
        ::"r"(tmem_d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrives once on bar when every tcgen05.mma this thread issued before it
// has completed (also when there is none).
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(saddr(bar)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Generic-proxy writes to shared memory made visible to the async proxy
// (the tensor cores read the converted A tiles through it).
__device__ __forceinline__ void fence_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Profiling hook: %globaltimer stamps of CTA 0 -- per chunk q < kTraceChunks
// 16 words: [0] producer issues, [1] converters see the stage, [2 + gi]
// converters release group gi, [6] MMA warp sees the stage, [7 + gi] MMAs of
// group gi issued, [11 + gi] epilogue sees group gi's accumulator, [15]
// epilogue releases the stage.
constexpr int kTraceChunks = 64;
__device__ __forceinline__ void trace_at(unsigned long long *tr, int q, int k) {
    if (tr != nullptr && blockIdx.x == 0 && (threadIdx.x & 31) == 0 && q < kTraceChunks && k < 16)
        tr[q * 16 + k] = globaltimer_ns();
}

__device__ __forceinline__ void epi_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
}

// TMEM loads: lane i of the warp gets TMEM lane (taddr >> 16) + i, columns
// (taddr & 0xffff) .. + n - 1; the wait is part of the statement, so the
// registers are complete when it ends.
__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_x64(uint32_t taddr, uint32_t (&r)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr)
        : "memory");
}

// Bounded wait of a whole warp (lane 0 polls) that also gives up as soon as
// another role has aborted; the first expiry records MOE_ETIMEOUT and raises
// the abort flag.  Every lane then observes the completed phase itself.
__device__ __forceinline__ bool uwait(uint64_t *bar, uint32_t parity, uint64_t timeout_ns,
                                      volatile int *abort_flag, int32_t *err) {
    // fast path: the phase has completed -- one probe by every lane
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    uint32_t ok = 0;
    if ((threadIdx.x & 31) == 0 && !*abort_flag) {
        ok = mbar_try_wait(bar, parity);
        const uint64_t t0 = ok ? 0 : globaltimer_ns();
        for (uint32_t i = 1; !ok; i++) {
            ok = mbar_try_wait(bar, parity);
            if (!ok && (i & 15) == 0) {
                if (*abort_flag) break;
                if (globaltimer_ns() - t0 > timeout_ns) {
                    atomicExch(err, MOE_ETIMEOUT);
                    *abort_flag = 1;
                    break;
                }
            }
        }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) mbar_try_wait(bar, parity);
    return ok != 0;
}

// One record's 64-column group of codes (this thread's row r of the stage)
// into row r of an A tile: 8 chunks of 8 bf16 values c + q, chunk j stored
// at 16 * (j ^ (r % 8)) (the 128-byte swizzle), so the 8 lanes of a
// store phase hit 8 different bank groups.
template <int BITS>
__device__ __forceinline__ void convert_row(const uint8_t *stage, int gi, uint8_t *tile, int r) {
    uint8_t *dst = tile + r * 128;
    if (BITS == 4) {
        // the record's 128-byte row holds the chunk's groups, 16-byte piece c
        // at 16 * (c ^ (r % 8)): the 8 lanes of a load phase read 8 different
        // bank groups
        const uint8_t *src = stage + r * 128;
#pragma unroll
        for (int h = 0; h < 2; h++) {
            const int c = 2 * gi + h;
            const uint4 w = *reinterpret_cast<const uint4 *>(src + ((c ^ (r & 7)) << 4));
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const uint32_t e = (ws[i] << 3) & 0x78787878u, o = (ws[i] >> 1) & 0x78787878u;
                uint4 out;
                out.x = pair_from(e, o, 0, 0x00780078u, 0x41804180u);
                out.y = pair_from(e, o, 1, 0x00780078u, 0x41804180u);
                out.z = pair_from(e, o, 2, 0x00780078u, 0x41804180u);
                out.w = pair_from(e, o, 3, 0x00780078u, 0x41804180u);
                const int j = 4 * h + i;
                *reinterpret_cast<uint4 *>(dst + ((j ^ (r & 7)) << 4)) = out;
            }
        }
    } else {
        const uint4 w = *reinterpret_cast<const uint4 *>(stage + gi * kCodeGroup + r * 16);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const uint32_t c0 = (ws[i] << 5) & 0x60606060u, c1 = (ws[i] << 3) & 0x60606060u;
            const uint32_t c2 = (ws[i] << 1) & 0x60606060u, c3 = (ws[i] >> 1) & 0x60606060u;
#pragma unroll
            for (int hb = 0; hb < 2; hb++) {
                const int b = 2 * hb;
                uint4 out;
                out.x = pair_from(c0, c1, b, 0x00600060u, 0x40804080u);
                out.y = pair_from(c2, c3, b, 0x00600060u, 0x40804080u);
                out.z = pair_from(c0, c1, b + 1, 0x00600060u, 0x40804080u);
                out.w = pair_from(c2, c3, b + 1, 0x00600060u, 0x40804080u);
                const int j = 2 * i + hb;
                *reinterpret_cast<uint4 *>(dst + ((j ^ (r & 7)) << 4)) = out;
            }
        }
    }
}

// Reads one group's accumulator (NC of its columns) for this thread's record
// and folds it into the running totals: total[t] += s * acc[t] + (b - c s)
// * xsum[t] (the same two fmaf per term as the register engine).
template <int NC, int BITS>
__device__ __forceinline__ void fold_group(uint32_t taddr, float sc, float bi, const float *xs,
                                           int gi, float (&total)[kTok]) {
    uint32_t acc[NC];
    if (NC == 16) tmem_ld_x16(taddr, reinterpret_cast<uint32_t (&)[16]>(acc));
    else if (NC == 32) tmem_ld_x32(taddr, reinterpret_cast<uint32_t (&)[32]>(acc));
    else tmem_ld_x64(taddr, reinterpret_cast<uint32_t (&)[64]>(acc));
    const float cb = fmaf(-pipe::CodeOff<BITS>::c, sc, bi);
#pragma unroll
    for (int t = 0; t < NC; t++)
        total[t] = fmaf(sc, __uint_as_float(acc[t]), fmaf(cb, xs[t * kGpc + gi], total[t]));
}

// The persistent kernel (the Job interface of gemm_pipe.cuh).
template <int BITS, class Job>
__global__ void __launch_bounds__(kThreads, 1) umma_gemm_kernel(const __grid_constant__ Job job,
                                                                const uint64_t timeout_ns,
                                                                const int stall,
                                                                unsigned long long *tr) {
    extern __shared__ __align__(1024) uint8_t smdyn[];
    uint8_t *stages = smdyn + ((1024u - (saddr(smdyn) & 1023u)) & 1023u);
    uint8_t *tiles = stages + kStages * kStageB;
    uint64_t *full = reinterpret_cast<uint64_t *>(tiles + kSlots * kSlotB);
    uint64_t *empty = full + kStages;
    uint64_t *a_full = empty + kStages, *a_empty = a_full + kBanks;
    uint64_t *acc_full = a_empty + kBanks, *acc_empty = acc_full + kBanks;
    uint64_t *stall_bar = acc_empty + kBanks;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(stall_bar + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
    int32_t *sm = reinterpret_cast<int32_t *>(tmem_holder + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; s++) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, kCvtWarps + 1 + kEpiWarps);
        }
        for (int k = 0; k < kBanks; k++) {
            mbar_init(a_full + k, kCvtWarps);
            mbar_init(a_empty + k, 1);
            mbar_init(acc_full + k, 1);
            mbar_init(acc_empty + k, kEpiWarps);
        }
        mbar_init(stall_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(saddr(tmem_holder)), "n"(kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    job.init(sm);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const int n_items = job.n_items(sm);
    const int b = blockIdx.x, nb = gridDim.x;
    const int mine = n_items > b ? (n_items - 1 - b) / nb + 1 : 0;
    const int nch = (job.cols + kKc - 1) / kKc;
    const int nq = mine * nch;
    int32_t *err = job.err;

    if (warp == kProdWarp) {
        // ------------------------------------------------ producer
        const uint64_t policy = pipe::evict_first_policy();
        const int cbytes = job.cols * BITS / 8;
        constexpr int kGB = kGroup * BITS / 8;       // code bytes of a group's row
        int li = 0, lc = 0, q = 0;
        Item it = nq > 0 ? job.item(sm, b) : Item{};
        for (; q < nq; q++) {
            const int s = q % kStages;
            uint8_t *stage = stages + s * kStageB;
            if (q >= kStages && !uwait(empty + s, ((q / kStages) - 1) & 1, timeout_ns, abort_flag, err))
                break;
            if (lc == nch - 1) {
                const int32_t *m = job.meta(sm, it);
                int32_t *ent = reinterpret_cast<int32_t *>(stage + kEntOff);
                if (m != nullptr)
                    for (int t = lane; t < it.nt; t += 32) ent[t] = m[t];
            }
            trace_at(tr, q < 32 ? q : 99, 0);
            // the chunk's copies: the codes (4-bit: one box; 2-bit: one per
            // group), the {s, b} words, per group the activation rows in one
            // box of 8, 16, 32 or 64 rows, their group sums -- each issued by
            // a lane of its own (one lane issues a copy every ~200 ns)
            const int ng = min(kKc, job.cols - lc * kKc) / kGroup;
            const int bk = it.nt <= 8 ? 0 : it.nt <= 16 ? 1 : it.nt <= 32 ? 2 : 3;
            const int rows = kRowBox << bk;
            const int ncodes = BITS == 4 ? 1 : ng;
            if (lane == 0)
                mbar_expect_tx(full + s, (BITS == 4 ? kRB * 128 : ng * kRB * kGB) + kRB * 16 +
                                             ng * rows * 128 + rows * 16);
            __syncwarp();
            int map, row, blob;
            job.weights(it, map, row, blob);
            const int r0 = job.row0(sm, it);
            if (lane < ncodes) {
                if (BITS == 4)
                    tma_3d(stage, &job.maps.gcodes[map], lc * kKc * BITS / 8, row, blob, full + s, policy);
                else
                    tma_3d(stage + lane * kCodeGroup, &job.maps.gcodes[map], (lc * kKc + lane * kGroup) * BITS / 8,
                           row, blob, full + s, policy);
            } else if (lane == ncodes) {
                tma_3d(stage + kSbOff, &job.maps.sb[map], cbytes + 16 * lc, row, blob, full + s, policy);
            } else if (lane < ncodes + 1 + ng) {
                const int gi = lane - ncodes - 1;
                tma_2d(stage + kXOff + gi * kXGroup, &job.maps.act128[bk], lc * kKc + gi * kGroup, r0, full + s);
            } else if (lane == ncodes + 1 + ng) {
                tma_2d(stage + kXsOff, &job.maps.gsum4[bk], lc * kGpc, r0, full + s);
            }
            if (++lc == nch) {
                lc = 0;
                if (++li < mine) it = job.item(sm, b + li * nb);
            }
        }
        // the copies of the last fill of each stage land before the CTA exits
        for (int s = 0; s < kStages && s < q; s++) {
            const int last = q - 1 - ((q - 1 - s) % kStages);
            if (!pipe::warp_wait(full + s, (last / kStages) & 1, timeout_ns) && lane == 0)
                atomicExch(err, MOE_ETIMEOUT);
        }
    } else if (warp >= kEpiWarps && warp < kMmaWarp) {
        // ------------------------------------------------ converters
        const int r = threadIdx.x - kEpiWarps * 32;
        int g = 0, lc = 0;
        for (int q = 0; q < nq; q++) {
            const int s = q % kStages;
            const uint8_t *stage = stages + s * kStageB;
            const bool have = uwait(full + s, (q / kStages) & 1, timeout_ns, abort_flag, err);
            if (warp == kEpiWarps) trace_at(tr, q < 32 ? q : 99, 1);
            const int ng = min(kKc, job.cols - lc * kKc) / kGroup;
            bool free = true;
            for (int gi = 0; gi < ng; gi++, g++) {
                // bank (g / kPer) % kBanks of slots: one wait before its first
                // group, one release after its last
                const int k = g % kSlots, bank = (g / kPer) % kBanks, buse = g / kSlots;
                if (g % kPer == 0)
                    free = buse == 0 || uwait(a_empty + bank, (buse - 1) & 1, timeout_ns, abort_flag, err);
                if (have && free && !*abort_flag)
                    convert_row<BITS>(stage, gi, tiles + k * kSlotB, r);
                if (g % kPer == kPer - 1) {
                    fence_async_shared();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(a_full + bank);
                }
                if (warp == kEpiWarps) trace_at(tr, q < 32 ? q : 99, 2 + (gi & 3));
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty + s);
            if (++lc == nch) lc = 0;
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------ MMA issue
        int g = 0, lc = 0, li = 0;
        Item it = nq > 0 ? job.item(sm, b) : Item{};
        for (int q = 0; q < nq; q++) {
            const int s = q % kStages;
            const uint8_t *stage = stages + s * kStageB;
            const bool have = uwait(full + s, (q / kStages) & 1, timeout_ns, abort_flag, err);
            trace_at(tr, q < 32 ? q : 99, 6);
            const int ng = min(kKc, job.cols - lc * kKc) / kGroup;
            const int n = min(kTok, max(16, (it.nt + 15) / 16 * 16));
            const uint32_t idesc = idesc_bf16_m128(n);
            // a bank at a time: its groups' MMAs interleaved by K step, so that
            // consecutive MMAs accumulate into different TMEM tiles
            for (int gi0 = 0; gi0 < ng; gi0 += kPer, g += kPer) {
                const int bank = (g / kPer) % kBanks, buse = g / kSlots;
                if (g < 64) trace_at(tr, 32 + g / 4, (g % 4) * 4 + 0);
                const bool a_ok = uwait(a_full + bank, buse & 1, timeout_ns, abort_flag, err);
                if (g < 64) trace_at(tr, 32 + g / 4, (g % 4) * 4 + 1);
                const bool d_ok = buse == 0 || uwait(acc_empty + bank, (buse - 1) & 1, timeout_ns, abort_flag, err);
                tc_fence_after();
                if (g < 64) trace_at(tr, 32 + g / 4, (g % 4) * 4 + 2);
                if (lane == 0) {
                    if (have && a_ok && d_ok && !*abort_flag) {
                        uint64_t ad[kPer], bd[kPer];
#pragma unroll
                        for (int j = 0; j < kPer; j++) {
                            ad[j] = sw128_desc(saddr(tiles + ((g + j) % kSlots) * kSlotB));
                            bd[j] = sw128_desc(saddr(stage + kXOff + (gi0 + j) * kXGroup));
                        }
#pragma unroll
                        for (int kk = 0; kk < 4; kk++)      // K = 16 bf16 = 32 bytes per step
#pragma unroll
                            for (int j = 0; j < kPer; j++)
                                umma_bf16(tmem + ((g + j) % kSlots) * kAccCols, ad[j] + 2 * kk, bd[j] + 2 * kk,
                                          idesc, kk > 0);
                    }
                    if (g < 64) trace_at(tr, 32 + g / 4, (g % 4) * 4 + 3);
                    umma_commit(a_empty + bank);
                    umma_commit(acc_full + bank);
                }
                trace_at(tr, q < 32 ? q : 99, 7 + (gi0 & 3));
                __syncwarp();
            }
            if (lane == 0) umma_commit(empty + s);
            __syncwarp();
            if (++lc == nch) {
                lc = 0;
                if (++li < mine) it = job.item(sm, b + li * nb);
            }
        }
    } else {
        // ------------------------------------------------ epilogue
        const int r = threadIdx.x;                           // record of the item, TMEM lane
        const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
        if (stall && blockIdx.x == 0 && warp == 0) {
            // test hook: 16 bytes that no copy sends; the wait runs out and
            // the launch takes its expiry path
            if (lane == 0) mbar_expect_tx(stall_bar, 16);
            __syncwarp();
            uwait(stall_bar, 0, timeout_ns, abort_flag, err);
        }
        float total[kTok];
#pragma unroll
        for (int t = 0; t < kTok; t++) total[t] = 0.0f;
        int g = 0, lc = 0, li = 0;
        Item it = nq > 0 ? job.item(sm, b) : Item{};
        for (int q = 0; q < nq; q++) {
            const int s = q % kStages;
            uint8_t *stage = stages + s * kStageB;
            const bool have = uwait(full + s, (q / kStages) & 1, timeout_ns, abort_flag, err);
            const int ng = min(kKc, job.cols - lc * kKc) / kGroup;
            const int n = min(kTok, max(16, (it.nt + 15) / 16 * 16));
            const uint32_t *sbw = reinterpret_cast<const uint32_t *>(stage + kSbOff);
            const float *xs = reinterpret_cast<const float *>(stage + kXsOff);
            bool ok = true;
            for (int gi = 0; gi < ng; gi++, g++) {
                const int k = g % kSlots, bank = (g / kPer) % kBanks, buse = g / kSlots;
                if (g % kPer == 0) {
                    ok = uwait(acc_full + bank, buse & 1, timeout_ns, abort_flag, err);
                    tc_fence_after();
                }
                if (warp == 0) trace_at(tr, q < 32 ? q : 99, 11 + (gi & 3));
                // tcgen05.ld is warp-collective: the whole warp takes lane 0's view
                // of the abort flag
                const bool go = __shfl_sync(0xffffffffu, (int)(have && ok && !*abort_flag), 0) != 0;
                if (go) {
                    const float2 sb = sb_f(sbw[r * kGpc + gi]);
                    const uint32_t ta = lane_addr + k * kAccCols;
                    if (n <= 16) fold_group<16, BITS>(ta, sb.x, sb.y, xs, gi, total);
                    else if (n <= 32) fold_group<32, BITS>(ta, sb.x, sb.y, xs, gi, total);
                    else fold_group<64, BITS>(ta, sb.x, sb.y, xs, gi, total);
                }
                if (g % kPer == kPer - 1) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(acc_empty + bank);
                }
            }
            if (lc == nch - 1) {
                // the item's results: staged over this stage's activations
                // and sums (every group's MMAs have completed and every
                // epilogue warp has folded them), then the job's epilogue
                float *out = reinterpret_cast<float *>(stage + kXOff);
                epi_sync();
#pragma unroll
                for (int t = 0; t < kTok; t++)
                    if (t < it.nt) out[r * kOutLd + t] = total[t];
                epi_sync();
                if (!*abort_flag)
                    job.epilogue(sm, it, out, reinterpret_cast<const int32_t *>(stage + kEntOff), r,
                                 kEpiWarps * 32);
                epi_sync();
#pragma unroll
                for (int t = 0; t < kTok; t++) total[t] = 0.0f;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty + s);
            if (warp == 0) trace_at(tr, q < 32 ? q : 99, 15);
            if (++lc == nch) {
                lc = 0;
                if (++li < mine) it = job.item(sm, b + li * nb);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols)
                     : "memory");
    }
}

// The profiling hook's buffer (device, kTraceChunks * 16 words) or null.
inline unsigned long long *&trace_buf() {
    static unsigned long long *p = nullptr;
    return p;
}

// Launches the kernel on every SM.  scratch_bytes: the job's shared scratch.
template <int BITS, class Job>
inline int launch_umma_gemm(const Job &job, size_t scratch_bytes, int sms, cudaStream_t st,
                            const char *name) {
    const size_t smem = kFixedSmem + scratch_bytes;
    cudaFuncSetAttribute(umma_gemm_kernel<BITS, Job>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
    const pipe::WaitCfg w = pipe::wait_cfg();
    umma_gemm_kernel<BITS, Job><<<sms, kThreads, smem, st>>>(
        job, w.timeout_ns ? w.timeout_ns : pipe::kDefaultWaitNs, w.stall, trace_buf());
    trace_buf() = nullptr;                 // the hook covers one launch
    return check_launch(name);
}

}  // namespace umma
}  // namespace moe

namespace moe {
namespace umma {

// Which engine runs a batched job, process-wide: 0 (default) and 1 = the
// register engine of gemm_pipe.cuh (mma.sync), 2 = this engine.  Measured on
// GB300 over T = 8 .. 4096 tokens of the 35B-like layer, this engine is 1.3x
// to 1.5x slower than the register engine at every size (the per-64-column
// affine fold keeps N at the item's <= 64 tokens, so its MMAs are small and
// their issue and hand-offs bound it), so the default stays the register
// engine.
inline int &engine_mode() {
    static int m = 0;
    return m;
}

template <int BITS, class Job>
inline int launch_batched_gemm(const Job &job, size_t scratch_bytes, int sms, cudaStream_t st,
                               const char *name, double mean_tokens) {
    const int mode = engine_mode();
    int dev = 0, smem_max = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    // the tensor-memory engine when its shared memory fits (the job's scratch
    // grows with the experts per layer)
    // (and the job's chunks hold whole banks: columns a multiple of kPer groups)
    const bool fits = kFixedSmem + scratch_bytes <= (size_t)smem_max && job.cols % (kPer * kGroup) == 0;
    (void)mean_tokens;
    const bool tc = fits && mode == 2;
    return tc ? launch_umma_gemm<BITS>(job, scratch_bytes, sms, st, name)
              : pipe::launch_pipe_gemm<BITS>(job, scratch_bytes, sms, st, name);
}

}  // namespace umma
}  // namespace moe
