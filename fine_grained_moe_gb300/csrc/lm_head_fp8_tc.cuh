// FP8 lm_head with argmax on the 5th-generation tensor cores (tcgen05).
//
//   z_{t,v} = scale[v] * sum_j e4m3(q[v][j]) h[t][j],   argmax over v per token
//
// The same product as k_lmhead_fp8 (lm_head_fp8.cuh), organised the sm_100
// way ("llm-decoding", §"Lever 1: fewer bytes (FP8 weights)": every weight in
// 8 bits; §"First principles": the tied lm_head is the largest matrix):
//  * One CTA per SM owns a contiguous range of 128-row vocabulary tiles.
//    (Ranges by rows, with the partial tile in 16-row boxes, balanced the
//    CTAs to 0.1 % instead of 4 % and ran 1.2 % slower: the copies, not the
//    balance, set the pace.)
//  * A producer thread streams each tile with TMA tensor copies
//    (cp.async.bulk.tensor.2d, 128 rows x 128 bytes, 128-byte swizzle) into a
//    5-stage ring of 32 KB stages (two K-chunks per stage), completing on
//    mbarriers. Rows past V come back as zeros.
//  * An MMA thread issues tcgen05.mma kind::f8f6f4, M = 128, N = 16, K = 32
//    (E4M3 x E4M3, fp32 accumulation) with both operands in shared memory:
//    A = the tile (K-major, swizzled by the copy), B = the hidden rows as two
//    E4M3 terms per value (column 2t + e = term e of token t), written once by
//    the CTA in the same swizzled K-major layout. The full-K accumulator of a
//    tile (128 lanes x 16 columns fp32) stays in tensor memory; two of them
//    alternate, so the next tile's products overlap this tile's epilogue.
//    tcgen05.commit frees a ring stage when its products are done.
//  * Four epilogue warps read their 32 lanes (rows) with tcgen05.ld, combine
//    the two terms, unscale (2^-s), apply the row scale and keep a running
//    (max, lowest index) per token; then a warp and CTA reduction gives one
//    partial per CTA, and the last CTA to finish reduces the partials and
//    applies greedy acceptance (as in k_lmhead_fp8).
//  * Hidden rows: each token is scaled by 2^s putting its largest |h| in
//    [2^7, 2^8); t0 = e4m3(y), t1 = e4m3(16 (y - t0)) hold a bf16 y exactly
//    while t1 stays normal (|y| above 2^-13 of the row maximum).
//  * NORM: the input is bf16(RMSNorm(h)) of the fp32 residual stream.
// Every wait is bounded (the library's wait limit); a timeout raises
// FGM_STATUS_WAIT_TIMEOUT, every role stops, the MMA thread waits for its
// issued products and the producer for its issued copies before the tensor
// memory is released and the CTA exits.
#pragma once

#include <cuda.h>

#include "basic_kernels.cuh"
#include "common.cuh"

namespace fgm {
namespace fp8tc {

constexpr int kThreads = 192;           // warp 0 producer, warp 1 MMA + TMEM owner, warps 2..5 epilogue
constexpr int kRows = 128;              // vocabulary rows per tile (the MMA's M)
constexpr int kN = 16;                  // MMA N: 8 tokens x 2 terms
constexpr int kChunk = 128;             // K bytes per TMA box and swizzle row
constexpr int kChunks = kH / kChunk;    // 22 K-chunks per row
constexpr int kChunksPerStage = 2;
constexpr int kStagesPerTile = kChunks / kChunksPerStage;   // 11
constexpr int kStages = 5;              // ring depth
constexpr int kBoxBytes = kRows * kChunk;                   // 16 KB
constexpr int kStageBytes = kChunksPerStage * kBoxBytes;    // 32 KB
constexpr int kBBytes = kChunks * kN * kChunk;              // 44 KB: B operand, 22 chunks of 16 rows x 128 B
constexpr int kRingOff = 0;
constexpr int kBOff = kStages * kStageBytes;                // 160 KB
constexpr int kSmemBytes = kBOff + kBBytes + 1024;          // + alignment slack to 1024 B
constexpr uint32_t kTmemCols = 32;                          // two 16-column accumulators
static_assert(kH % (kChunk * kChunksPerStage) == 0, "K must split into whole stages");

// tcgen05 instruction descriptor, kind::f8f6f4: D fp32 (bits 4-5 = 1), A and B
// E4M3 (format 0), both K-major, N >> 3 at bits 17-22, M >> 4 at bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (static_cast<uint32_t>(kN >> 3) << 17) | (static_cast<uint32_t>(kRows >> 4) << 24);

// Shared-memory matrix descriptor of a K-major operand in the 128-byte swizzle
// layout: 8-row x 128-byte atoms, 1024 bytes apart (stride byte offset);
// start address in 16-byte units; descriptor version 1; layout type 2.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr)
{
    return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) | (1ull << 16) | (64ull << 32) | (1ull << 46) |
           (2ull << 61);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ long long gtime()
{
    long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Arguments of one launch (the tensor map is a separate __grid_constant__).
struct Args {
    const float *scale;     // [V] row scales
    int V;
    const void *h;          // bf16 [M][2816] rows, or (NORM) the fp32 residual stream [M][2816]
    int M;
    float *part_val;        // [gridDim.x][8]
    int32_t *part_idx;      // [gridDim.x][8]
    unsigned *done;         // CTAs finished; 0 between launches (the last CTA resets it)
    int32_t *argmax;        // [M] output
    float *maxlogit;        // [M] output or NULL
    const int32_t *draft;   // [M - 1] drafts (used when out != NULL)
    int32_t *out;           // [2] {accepted, next} or NULL
    int32_t *status;        // FGM_STATUS_* bits
    long long timeout_ns;   // bound of every wait
};

struct Shared {
    unsigned long long full[kStages], empty[kStages], tfull[2], tempty[2], mma_done;
    uint32_t tmem_base;
    int abort;
    float rn[kMaxM];
    unsigned amax_bits[kMaxM];
    float up[kMaxM], down[kMaxM];
    float rv[4][kMaxM];
    int32_t ri[4][kMaxM];
    int32_t arg[kMaxM];
    int last;
};

// Byte offset of element (row n, k) of a K-major operand with 128-byte rows
// per chunk in the 128-byte swizzle: 16-byte unit (k % 128) / 16 of row n is
// stored at unit ((k % 128) / 16) ^ (n % 8) of its 128-byte row.
__device__ __forceinline__ uint32_t b_offset(int n, int k)
{
    const int c = k >> 7, kk = k & 127;
    return static_cast<uint32_t>(c * (kN * kChunk) + (n >> 3) * 1024 + (n & 7) * 128 + (((kk >> 4) ^ (n & 7)) << 4) +
                                 (kk & 15));
}

template <bool NORM>
__global__ void __launch_bounds__(kThreads, 1) k_lmhead_fp8_tc(const __grid_constant__ CUtensorMap tmap, const Args p)
{
    extern __shared__ uint8_t dsm_raw[];
    __shared__ Shared sh;
    // 1024-byte aligned base (swizzle atoms)
    const uint32_t raw = smem_u32(dsm_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *dsm = dsm_raw + (base - raw);
    const uint32_t ring = base + kRingOff, bsm = base + kBOff;
    uint8_t *bgen = dsm + kBOff;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int M = p.M, V = p.V;
    const long long deadline = gtime() + p.timeout_ns;
    const int T = (V + kRows - 1) / kRows;
    const int t_begin = static_cast<int>((long long)T * blockIdx.x / gridDim.x);
    const int t_end = static_cast<int>((long long)T * (blockIdx.x + 1) / gridDim.x);
    const int n_tiles = t_end - t_begin;

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(smem_u32(&sh.full[i]), 1);
            mbar_init(smem_u32(&sh.empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&sh.tfull[i]), 1);
            mbar_init(smem_u32(&sh.tempty[i]), 4);
        }
        mbar_init(smem_u32(&sh.mma_done), 1);
        sh.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        // tensor memory for the two accumulators (one CTA per SM: always granted)
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&sh.tmem_base)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    __syncthreads();

    // bounded wait on an mbarrier phase; false on timeout or abort
    auto wait = [&](uint32_t bar, uint32_t parity) -> bool {
        for (int it = 0;; ++it) {
            if (mbar_try(bar, parity))
                return true;
            if ((it & 255) == 255) {
                if (*reinterpret_cast<volatile int *>(&sh.abort))
                    return false;
                if (gtime() > deadline) {
                    *reinterpret_cast<volatile int *>(&sh.abort) = 1;
                    atomicOr(p.status, FGM_STATUS_WAIT_TIMEOUT);
                    return false;
                }
            }
        }
    };

    // producer: the first ring stages stream in while the hidden rows are prepared
    uint32_t p_stage = 0;   // stages issued
    auto produce = [&](int ti, int ks) -> bool {
        const int slot = p_stage % kStages;
        const uint32_t full = smem_u32(&sh.full[slot]);
        if (p_stage >= kStages && !wait(smem_u32(&sh.empty[slot]), ((p_stage / kStages) - 1) & 1))
            return false;
        mbar_expect_tx(full, kStageBytes);
        const int y = (t_begin + ti) * kRows;
        // rows read once per step: evict-first in L2
        uint64_t pol;
        asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
#pragma unroll
        for (int b = 0; b < kChunksPerStage; ++b) {
            const uint32_t dst = ring + slot * kStageBytes + b * kBoxBytes;
            const int x = (ks * kChunksPerStage + b) * kChunk;
            asm volatile(
                "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
                "{%2, %3}], [%4], %5;" ::"r"(dst),
                "l"(reinterpret_cast<uint64_t>(&tmap)), "r"(x), "r"(y), "r"(full), "l"(pol)
                : "memory");
        }
        ++p_stage;
        return true;
    };
    const int total_stages = n_tiles * kStagesPerTile;
    if (warp == 0 && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap)) : "memory");
        for (int i = 0; i < kStages && i < total_stages; ++i)
            produce(i / kStagesPerTile, i % kStagesPerTile);
    }

    // hidden rows -> B operand (all threads)
    auto hval = [&](int tk, int k) -> float {
        if constexpr (NORM)
            return bf16_to_f32(f32_to_bf16(static_cast<const float *>(p.h)[(size_t)tk * kH + k] * sh.rn[tk]));
        else
            return bf16_to_f32(static_cast<const uint16_t *>(p.h)[(size_t)tk * kH + k]);
    };
    if constexpr (NORM) {
        for (int tk = warp; tk < M; tk += kThreads / 32) {
            const float *row = static_cast<const float *>(p.h) + (size_t)tk * kH;
            float ss = 0.0f;
            for (int k = lane; k < kH; k += 32)
                ss += row[k] * row[k];
            ss = warp_sum(ss);
            if (lane == 0)
                sh.rn[tk] = 1.0f / sqrtf(ss / static_cast<float>(kH) + kEps);
        }
        __syncthreads();
    }
    for (int tk = warp; tk < kMaxM; tk += kThreads / 32) {
        unsigned m = 0;
        if (tk < M)
            for (int k = lane; k < kH; k += 32) {
                const float a = fabsf(hval(tk, k));
                if (a < INFINITY)
                    m = max(m, __float_as_uint(a));
            }
        m = __reduce_max_sync(0xFFFFFFFFu, m);
        if (lane == 0)
            sh.amax_bits[tk] = m;
    }
    __syncthreads();
    if (tid < kMaxM) {
        // 2^s puts the largest |h| in [2^7, 2^8); a zero or subnormal maximum keeps s = 0
        const int ef = static_cast<int>(sh.amax_bits[tid] >> 23);
        int s = ef == 0 ? 0 : 134 - ef;
        s = min(126, s);
        sh.up[tid] = __uint_as_float(static_cast<unsigned>(127 + s) << 23);
        sh.down[tid] = __uint_as_float(static_cast<unsigned>(127 - s) << 23);
    }
    __syncthreads();
    // column n = 2 tk + e holds term e of token tk (zero for tk >= M), 4 bytes a thread step
    for (int i = tid; i < kMaxM * (kH / 4); i += kThreads) {
        const int tk = i / (kH / 4), k = 4 * (i - tk * (kH / 4));
        uint32_t w0 = 0, w1 = 0;
        if (tk < M) {
            float y[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                y[j] = hval(tk, k + j) * sh.up[tk];
            const __nv_fp8x2_storage_t a0 = __nv_cvt_float2_to_fp8x2(make_float2(y[0], y[1]), __NV_SATFINITE, __NV_E4M3);
            const __nv_fp8x2_storage_t a1 = __nv_cvt_float2_to_fp8x2(make_float2(y[2], y[3]), __NV_SATFINITE, __NV_E4M3);
            w0 = static_cast<uint32_t>(a0) | (static_cast<uint32_t>(a1) << 16);
            const float2 d0 = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(a0, __NV_E4M3)));
            const float2 d1 = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(a1, __NV_E4M3)));
            const __nv_fp8x2_storage_t b0 = __nv_cvt_float2_to_fp8x2(
                make_float2(16.0f * (y[0] - d0.x), 16.0f * (y[1] - d0.y)), __NV_SATFINITE, __NV_E4M3);
            const __nv_fp8x2_storage_t b1 = __nv_cvt_float2_to_fp8x2(
                make_float2(16.0f * (y[2] - d1.x), 16.0f * (y[3] - d1.y)), __NV_SATFINITE, __NV_E4M3);
            w1 = static_cast<uint32_t>(b0) | (static_cast<uint32_t>(b1) << 16);
        }
        *reinterpret_cast<uint32_t *>(bgen + b_offset(2 * tk, k)) = w0;
        *reinterpret_cast<uint32_t *>(bgen + b_offset(2 * tk + 1, k)) = w1;
    }
    // the B operand is read by the tensor cores (async proxy)
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    const uint32_t tmem = sh.tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            bool ok = true;
            for (int i = kStages; i < total_stages && ok; ++i)
                ok = produce(i / kStagesPerTile, i % kStagesPerTile);
            // every issued copy lands before the CTA may exit
            const uint32_t first = p_stage > kStages ? p_stage - kStages : 0;
            for (uint32_t k = first; k < p_stage; ++k)
                for (int it = 0; it < (1 << 22); ++it)
                    if (mbar_try(smem_u32(&sh.full[k % kStages]), (k / kStages) & 1))
                        break;
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            bool ok = true;
            uint32_t c_stage = 0;
            for (int ti = 0; ti < n_tiles && ok; ++ti) {
                const int buf = ti & 1;
                // the epilogue has read this accumulator two tiles ago
                if (ti >= 2 && !(ok = wait(smem_u32(&sh.tempty[buf]), ((ti >> 1) - 1) & 1)))
                    break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t d = tmem + static_cast<uint32_t>(buf * kN);
                for (int ks = 0; ks < kStagesPerTile && ok; ++ks, ++c_stage) {
                    const int slot = c_stage % kStages;
                    if (!(ok = wait(smem_u32(&sh.full[slot]), (c_stage / kStages) & 1)))
                        break;
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
                    for (int b = 0; b < kChunksPerStage; ++b)
#pragma unroll
                        for (int kk = 0; kk < kChunk / 32; ++kk) {
                            const uint64_t ad = smem_desc(ring + slot * kStageBytes + b * kBoxBytes + kk * 32);
                            const uint64_t bd =
                                smem_desc(bsm + (ks * kChunksPerStage + b) * (kN * kChunk) + kk * 32);
                            const uint32_t acc = (ks | b | kk) != 0;
                            asm volatile(
                                "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
                                "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
                                "l"(ad), "l"(bd), "r"(kIdesc), "r"(acc)
                                : "memory");
                        }
                    // the stage's slot is free once these products are done
                    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                                     smem_u32(&sh.empty[slot]))
                                 : "memory");
                }
                if (ok)
                    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                                     smem_u32(&sh.tfull[buf]))
                                 : "memory");
            }
            // every issued product completes before the tensor memory is released
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                             smem_u32(&sh.mma_done))
                         : "memory");
            for (int it = 0; it < (1 << 22); ++it)
                if (mbar_try(smem_u32(&sh.mma_done), 0))
                    break;
        }
        __syncwarp();
    }

    // ---------------------------------------------------------------- epilogue
    // warps 2..5 read TMEM lanes 32 (warp % 4) .. + 31: row r of each tile
    float bv[kMaxM];
    int32_t bi[kMaxM];
#pragma unroll
    for (int t = 0; t < kMaxM; ++t) {
        bv[t] = -INFINITY;
        bi[t] = 0x7FFFFFFF;
    }
    if (warp >= 2) {
        const int quarter = warp & 3;
        const int r = 32 * quarter + lane;
        for (int ti = 0; ti < n_tiles; ++ti) {
            const int buf = ti & 1;
            if (!wait(smem_u32(&sh.tfull[buf]), (ti >> 1) & 1))
                break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            uint32_t v[kN];
            const uint32_t ta = tmem + (static_cast<uint32_t>(32 * quarter) << 16) + static_cast<uint32_t>(buf * kN);
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
                "%14, %15}, [%16];"
                : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
                  "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
                : "r"(ta)
                : "memory");
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&sh.tempty[buf]));
            const int row = (t_begin + ti) * kRows + r;
            if (row < V) {
                const float s = __ldg(p.scale + row);
#pragma unroll
                for (int t = 0; t < kMaxM; ++t) {
                    if (t < M) {
                        const float z =
                            (__uint_as_float(v[2 * t]) + 0.0625f * __uint_as_float(v[2 * t + 1])) * sh.down[t] * s;
                        if (better(z, row, bv[t], bi[t])) {
                            bv[t] = z;
                            bi[t] = row;
                        }
                    }
                }
            }
        }
        // warp reduction per token, then one entry per epilogue warp
#pragma unroll
        for (int t = 0; t < kMaxM; ++t) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv[t], o);
                const int32_t oi = __shfl_xor_sync(0xFFFFFFFFu, bi[t], o);
                if (better(ov, oi, bv[t], bi[t])) {
                    bv[t] = ov;
                    bi[t] = oi;
                }
            }
            if (lane == 0) {
                sh.rv[warp - 2][t] = bv[t];
                sh.ri[warp - 2][t] = bi[t];
            }
        }
    }
    __syncthreads();
    if (warp == 1) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
    if (tid < M) {
        float v = sh.rv[0][tid];
        int32_t ix = sh.ri[0][tid];
        for (int w = 1; w < 4; ++w)
            if (better(sh.rv[w][tid], sh.ri[w][tid], v, ix)) {
                v = sh.rv[w][tid];
                ix = sh.ri[w][tid];
            }
        p.part_val[blockIdx.x * kMaxM + tid] = v;
        p.part_idx[blockIdx.x * kMaxM + tid] = ix;
    }

    // the last CTA to finish reduces every CTA's partial
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        sh.last = atomicAdd(p.done, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (!sh.last)
        return;
    __threadfence();
    for (int tk = warp; tk < M; tk += kThreads / 32) {
        float v = -INFINITY;
        int32_t ix = 0x7FFFFFFF;
        for (int c = lane; c < (int)gridDim.x; c += 32) {
            const float ov = __ldcg(p.part_val + c * kMaxM + tk);
            const int32_t oi = __ldcg(p.part_idx + c * kMaxM + tk);
            if (better(ov, oi, v, ix)) {
                v = ov;
                ix = oi;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xFFFFFFFFu, v, o);
            const int32_t oi = __shfl_xor_sync(0xFFFFFFFFu, ix, o);
            if (better(ov, oi, v, ix)) {
                v = ov;
                ix = oi;
            }
        }
        if (lane == 0) {
            if (ix == 0x7FFFFFFF) {   // every logit was NaN
                ix = 0;
                atomicOr(p.status, FGM_STATUS_NONFINITE_LOGITS);
            }
            sh.arg[tk] = ix;
            p.argmax[tk] = ix;
            if (p.maxlogit)
                p.maxlogit[tk] = v;
        }
    }
    __syncthreads();
    if (tid == 0) {
        if (p.out)
            accept_greedy(sh.arg, p.draft, M, p.out);
        *p.done = 0u;
    }
}

// CTAs for V rows: one per SM, fewer when there are not enough tiles.
inline int grid_for(int64_t V, int sms)
{
    const int64_t tiles = (V + kRows - 1) / kRows;
    const int64_t g = tiles < sms ? tiles : sms;
    return g < 1 ? 1 : static_cast<int>(g < kMaxParts ? g : kMaxParts);
}

}  // namespace fp8tc
}  // namespace fgm
