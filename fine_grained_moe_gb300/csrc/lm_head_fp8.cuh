// FP8 lm_head with argmax. The tied embedding is stored as E4M3 codes with one
// fp32 scale per vocabulary row (the format of the expert weights), which
// halves the bytes of the largest single matrix of the step: 0.74 GB instead
// of 1.48 GB for 262,144 x 2816 ("llm-decoding", §"Lever 1: fewer bytes (FP8
// weights)" stores every weight in 8 bits; §"First principles: compute-bound
// or memory-bound?" counts the BF16 projection at a fifth of a token's bytes).
//
//   z_{t,v} = scale[v] * sum_j e4m3(q[v][j]) h[t][j],   argmax over v per token
//
// Design (one pass over q at HBM speed):
//  * One CTA per SM, 16 warps. CTA b owns a contiguous range of whole 16-row
//    tiles of the vocabulary, T/G of them to within one (G CTAs), dealt to its
//    warps round-robin; each tile's 45 KB is read once. (Dealing tiles
//    round-robin over all warps of the grid left 112 SMs with 112 tiles and 40
//    with 96: the kernel is bound by per-SM MMA throughput, so that cost ~4%.) A lane copies 16 bytes of row g = lane / 4 and of row
//    g + 8 per 64-byte K-block, so four lanes cover 64 contiguous bytes of a
//    row and a warp step touches full 32-byte sectors only.
//  * Products on the tensor cores as E4M3 x E4M3: mma.sync m16n8k32 with
//    fp32 accumulation, the weight codes used as they are stored (no
//    conversion in the loop). The 8 MMA columns are the tokens (absent tokens
//    are zero). Within a K-block the lane's 16 bytes are two k32 slices:
//    bytes 0..3 and 4..7 are the A fragment's k 4t..4t+3 and 4t+16..4t+19 of
//    slice 0, bytes 8..15 those of slice 1; the B fragment maps k the same way
//    (it depends on t only), so every product meets its own hidden element.
//  * The hidden rows live in shared memory as two E4M3 terms per value. Each
//    token is scaled by a power of two 2^s that puts its largest |h| in
//    [2^7, 2^8); then t0 = e4m3(y) and t1 = e4m3(16 (y - t0)) represent a bf16
//    y exactly (8 significant bits = 4 + 4) over the 2^13 below the maximum
//    that matter. The two terms are two accumulators, combined and unscaled
//    (exactly, by 2^-s) in the epilogue. A conversion of each weight to f16
//    for an f16 MMA instead kept the ALU pipe half busy and the kernel at
//    0.86 of the copy bandwidth.
//  * Copies run through a per-warp ring in shared memory: each lane issues
//    cp.async (L1 bypassed) for its own bytes kDepth - 1 = 4 steps of 2 KB
//    per warp ahead of the products, across tile boundaries too, so 128 KB
//    per SM is in flight without holding registers (a register double buffer
//    held 64 KB and left the loads latency-bound).
//  * Epilogue per tile: row scale, unscale, running (max, lowest index) per
//    token; then a warp and CTA reduction to one partial per CTA. The last
//    CTA to finish (a completion count in the workspace) reduces the
//    partials and applies greedy acceptance, so a call is one launch.
//  * For the verify step the kernel also applies the final unit RMSNorm to
//    the fp32 residual stream in its prologue (NORM), while the first ring
//    stages are already streaming in.
#pragma once

#include "basic_kernels.cuh"
#include "common.cuh"

namespace fgm {
namespace fp8head {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kRows = 16;                  // vocabulary rows per warp tile (the MMA's M)
constexpr int kTerms = 2;                  // E4M3 terms per hidden value (exact for bf16 inputs)
constexpr int kColPitch = kH + 64;         // bytes per (term, token) column in shared memory: a 64-byte
                                           // offset between neighbouring tokens keeps B loads conflict-free
constexpr int kBlock = 64;                 // K bytes per lane quad and K-block (4 lanes x 16 bytes)
constexpr int kBlocks = kH / kBlock;       // 44 K-blocks per row
constexpr int kGroup = 2;                  // K-blocks per pipeline step
constexpr int kSteps = kBlocks / kGroup;   // 22 steps per tile
constexpr int kDepth = 5;                  // ring stages per warp (kDepth - 1 steps in flight)
constexpr int kStageVecs = 2 * kGroup * 32;                      // 16-byte vectors per stage (2 KB)
constexpr int kHsBytes = kTerms * kMaxM * kColPitch;             // hidden-row terms
constexpr int kSmemBytes = kHsBytes + kWarps * kDepth * kStageVecs * 16;  // dynamic shared memory
static_assert(kH % (kBlock * kGroup) == 0, "hidden width must split into whole pipeline steps");
static_assert(kHsBytes % 16 == 0 && kColPitch % 128 == 64, "column layout");

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16 bytes global -> shared, bypassing L1; L2 fetches the surrounding 256 bytes
// and marks them evict-first: the rows are read once per step, and the small
// data that the next launch reads again stays in L2.
__device__ __forceinline__ void cp_async16(uint32_t dst, const uint8_t *src)
{
    uint64_t pol;
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    asm volatile("cp.async.cg.shared.global.L2::cache_hint.L2::256B [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "l"(pol)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// D += A (16 x 32, E4M3, row-major) x B (32 x 8, E4M3), fp32 accumulation.
__device__ __forceinline__ void mma_e4m3(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Nearest E4M3 codes of two floats (low byte = a), saturating at +-448.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float a, float b)
{
    return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

// The value of an E4M3 code pair as two floats (exact).
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t two)
{
    const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two & 0xFFFFu), __NV_E4M3);
    return __half22float2(__half2(r));
}

// Arguments of one launch.
struct Args {
    const uint8_t *q;       // [V][2816] E4M3 codes
    const float *scale;     // [V] row scales
    int V;
    const void *h;          // bf16 [M][2816] rows, or (NORM) the fp32 residual stream [M][2816]
    int M;
    float *part_val;        // [gridDim.x][8] per-CTA best logit
    int32_t *part_idx;      // [gridDim.x][8] and its row
    unsigned *done;         // CTAs finished; 0 between launches (the last CTA resets it)
    int32_t *argmax;        // [M] output
    float *maxlogit;        // [M] output or NULL
    const int32_t *draft;   // [M - 1] drafts (used when out != NULL)
    int32_t *out;           // [2] {accepted, next} or NULL
    int32_t *status;        // FGM_STATUS_* bits
};

// One pass over the E4M3 rows: per-CTA argmax partials, then the last CTA to
// finish reduces them (ties to the lower row) and, with `out`, applies greedy
// acceptance. NORM: the lm_head input is bf16(RMSNorm(h)) of the fp32 rows
// (unit gain, eps 1e-6), else the given bf16 rows.
template <bool NORM>
__global__ void __launch_bounds__(kThreads, 1) k_lmhead_fp8(const Args p)
{
    extern __shared__ __align__(16) uint8_t dsm[];          // [kHsBytes] hidden rows, then the rings
    uint8_t *hs = dsm;   // [term][token][kColPitch] E4M3 terms of h * 2^s, zero for tokens >= M
    __shared__ float rn[kMaxM];                              // NORM: 1 / rms of each row
    __shared__ unsigned amax_bits[kMaxM];
    __shared__ float up[kMaxM], down[kMaxM];                 // 2^s and 2^-s per token
    __shared__ float rv[kWarps][kMaxM];
    __shared__ int32_t ri[kWarps][kMaxM];
    __shared__ int32_t s_arg[kMaxM];
    __shared__ int s_last;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int M = p.M, V = p.V;
    const uint8_t *__restrict__ q = p.q;

    // Ring of this warp: kDepth stages. A stage is one pipeline step of the
    // warp's current tile: per lane kGroup K-blocks of rows g and g + 8, 16
    // bytes each, copied by the lane itself with cp.async; chunk j = 2 b +
    // (row g + 8) of lane l sits at ring[stage][j][l], so the lane's copies
    // and loads are conflict-free. Each lane reads back only its own copies,
    // so the wait on its own commit groups is all a stage needs.
    const int T = (V + kRows - 1) / kRows;
    // this CTA's tiles: a contiguous range of floor or ceil(T / CTAs), dealt to
    // its warps round-robin (the SMs, not the warps, share the bandwidth)
    const int t_begin = static_cast<int>((long long)T * blockIdx.x / gridDim.x);
    const int t_end = static_cast<int>((long long)T * (blockIdx.x + 1) / gridDim.x);
    const uint4 *ring = reinterpret_cast<const uint4 *>(dsm + kHsBytes) + (size_t)warp * kDepth * kStageVecs;
    const uint32_t ring_lane = smem_u32(ring + lane);
    // rows g and g + 8 of tile tl (rows past the end read row V - 1 and are dropped)
    auto row_ptrs = [&](int tl, const uint8_t *&pa, const uint8_t *&pb) {
        const int r0 = min(tl * kRows + g, V - 1), r1 = min(tl * kRows + g + 8, V - 1);
        pa = q + (size_t)r0 * kH + 16 * t;
        pb = q + (size_t)r1 * kH + 16 * t;
    };
    // issue side: tile `it`, step `is` of the next stage to copy; once past the
    // last tile it commits empty groups, so the wait below counts uniformly
    int it = t_begin + warp, is = 0;
    const uint8_t *ia = q, *ib = q;
    if (it < t_end)
        row_ptrs(it, ia, ib);
    auto issue = [&](int slot) {
        if (it < t_end) {
            const uint32_t dst = ring_lane + static_cast<uint32_t>(slot * kStageVecs) * 16u;
#pragma unroll
            for (int b = 0; b < kGroup; ++b) {
                cp_async16(dst + (2 * b) * 32 * 16, ia + (is * kGroup + b) * kBlock);
                cp_async16(dst + (2 * b + 1) * 32 * 16, ib + (is * kGroup + b) * kBlock);
            }
            if (++is == kSteps) {
                is = 0;
                it += kWarps;
                if (it < t_end)
                    row_ptrs(it, ia, ib);
            }
        }
        cp_async_commit();
    };
    // the first stages stream in while the hidden rows are prepared
#pragma unroll
    for (int d = 0; d < kDepth - 1; ++d)
        issue(d);

    // lm_head input elements 2 k2, 2 k2 + 1 of token tk (tk < M)
    auto hval2 = [&](int tk, int k2) -> float2 {
        if constexpr (NORM) {
            const float2 v = *reinterpret_cast<const float2 *>(static_cast<const float *>(p.h) + (size_t)tk * kH + 2 * k2);
            return make_float2(bf16_to_f32(f32_to_bf16(v.x * rn[tk])), bf16_to_f32(f32_to_bf16(v.y * rn[tk])));
        } else {
            return bf16x2_to_f32(*reinterpret_cast<const uint32_t *>(static_cast<const uint16_t *>(p.h) +
                                                                     (size_t)tk * kH + 2 * k2));
        }
    };
    // 1. NORM: 1 / sqrt(mean(h^2) + eps) per token
    if constexpr (NORM) {
        for (int tk = warp; tk < M; tk += kWarps) {
            const float *row = static_cast<const float *>(p.h) + (size_t)tk * kH;
            float ss = 0.0f;
            for (int k = lane; k < kH; k += 32)
                ss += row[k] * row[k];
            ss = warp_sum(ss);
            if (lane == 0)
                rn[tk] = 1.0f / sqrtf(ss / static_cast<float>(kH) + kEps);
        }
        __syncthreads();
    }
    // 2. largest finite |input| per token (non-negative floats order like their bits)
    for (int tk = warp; tk < kMaxM; tk += kWarps) {
        unsigned m = 0;
        if (tk < M)
            for (int k2 = lane; k2 < kH / 2; k2 += 32) {
                const float2 v = hval2(tk, k2);
                const float a = fabsf(v.x), b = fabsf(v.y);
                if (a < INFINITY)
                    m = max(m, __float_as_uint(a));
                if (b < INFINITY)
                    m = max(m, __float_as_uint(b));
            }
        m = __reduce_max_sync(0xFFFFFFFFu, m);
        if (lane == 0)
            amax_bits[tk] = m;
    }
    __syncthreads();
    // 3. s = 134 - biased exponent of that max puts it in [2^7, 2^8), below
    //    E4M3's 448; a zero or subnormal max keeps s = 0. For finite maxima
    //    s >= -120; s <= 126 keeps 2^s and 2^-s normal floats
    if (tid < kMaxM) {
        const int ef = static_cast<int>(amax_bits[tid] >> 23);
        int s = ef == 0 ? 0 : 134 - ef;
        s = min(126, s);
        up[tid] = __uint_as_float(static_cast<unsigned>(127 + s) << 23);
        down[tid] = __uint_as_float(static_cast<unsigned>(127 - s) << 23);
    }
    __syncthreads();
    // 4. y = input * 2^s as two E4M3 terms, y = t0 + t1 / 16 with t0 = e4m3(y)
    //    and t1 = e4m3(16 (y - t0)). A bf16 y has 8 significant bits, t0 holds
    //    the top 4 and the remainder is a 4-bit multiple of y's ulp, so t1
    //    holds it exactly while it stays in E4M3's normal range (|y| above
    //    max * 2^-13; smaller values lose low bits, below 2^-13 of the row's
    //    largest product)
    for (int i = tid; i < kMaxM * (kH / 2); i += kThreads) {
        const int tk = i / (kH / 2), k2 = i - tk * (kH / 2);
        uint32_t w0 = 0, w1 = 0;
        if (tk < M) {
            const float2 v = hval2(tk, k2);
            const float y0 = v.x * up[tk], y1 = v.y * up[tk];
            w0 = f32x2_to_e4m3x2(y0, y1);
            const float2 d = e4m3x2_to_f32x2(w0);
            w1 = f32x2_to_e4m3x2(16.0f * (y0 - d.x), 16.0f * (y1 - d.y));
        }
        *reinterpret_cast<uint16_t *>(hs + tk * kColPitch + 2 * k2) = static_cast<uint16_t>(w0);
        *reinterpret_cast<uint16_t *>(hs + (kMaxM + tk) * kColPitch + 2 * k2) = static_cast<uint16_t>(w1);
    }
    __syncthreads();

    // 5. stream the tiles through the ring
    const uint8_t *hrow = hs + g * kColPitch + 16 * t;   // B operand: token g, this lane's 16 k per block
    const float *__restrict__ scale = p.scale;
    float bv[2] = {-INFINITY, -INFINITY};               // tokens 2t, 2t + 1
    int32_t bi[2] = {0x7FFFFFFF, 0x7FFFFFFF};

    int slot = 0;
    for (int tile = t_begin + warp; tile < t_end; tile += kWarps) {
        const int r0 = tile * kRows + g, r1 = r0 + 8;
        const float s0 = scale[min(r0, V - 1)], s1 = scale[min(r1, V - 1)];
        float c[kTerms][4] = {};   // per term: row g tokens 2t, 2t + 1; row g + 8 the same
#pragma unroll
        for (int s = 0; s < kSteps; ++s) {
            issue(slot == 0 ? kDepth - 1 : slot - 1);   // the stage consumed last (its reads are done)
            cp_async_wait<kDepth - 1>();                // this lane's copies of stage `slot` landed
            const uint4 *st = ring + slot * kStageVecs + lane;
#pragma unroll
            for (int b = 0; b < kGroup; ++b) {
                const int kb = s * kGroup + b;
                // bytes 0..7 of the lane's chunk are k32 slice 0 (A words x, y:
                // k 4t..4t+3 and 4t+16..4t+19 of the MMA), bytes 8..15 slice 1;
                // the B words of each term follow the same map
                const uint4 va = st[(2 * b) * 32], vb = st[(2 * b + 1) * 32];
                const uint4 h0 = *reinterpret_cast<const uint4 *>(hrow + kb * kBlock);
                const uint4 h1 = *reinterpret_cast<const uint4 *>(hrow + kMaxM * kColPitch + kb * kBlock);
                mma_e4m3(c[0], va.x, vb.x, va.y, vb.y, h0.x, h0.y);
                mma_e4m3(c[1], va.x, vb.x, va.y, vb.y, h1.x, h1.y);
                mma_e4m3(c[0], va.z, vb.z, va.w, vb.w, h0.z, h0.w);
                mma_e4m3(c[1], va.z, vb.z, va.w, vb.w, h1.z, h1.w);
            }
            slot = slot + 1 == kDepth ? 0 : slot + 1;
        }
        // c[e][u]: row r0, token 2t + u; c[e][2 + u]: row r1, token 2t + u
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int tk = 2 * t + u;
            if (tk < M) {
                const float dn = down[tk];
                if (r0 < V) {
                    const float z = (c[0][u] + c[1][u] * 0.0625f) * s0 * dn;
                    if (better(z, r0, bv[u], bi[u])) {
                        bv[u] = z;
                        bi[u] = r0;
                    }
                }
                if (r1 < V) {
                    const float z = (c[0][2 + u] + c[1][2 + u] * 0.0625f) * s1 * dn;
                    if (better(z, r1, bv[u], bi[u])) {
                        bv[u] = z;
                        bi[u] = r1;
                    }
                }
            }
        }
    }
    cp_async_wait<0>();   // nothing of this lane may be in flight when the CTA exits

    // 6. this CTA's partial: warp (lanes of equal t), then CTA
#pragma unroll
    for (int o = 4; o < 32; o <<= 1)
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv[u], o);
            const int32_t oi = __shfl_xor_sync(0xFFFFFFFFu, bi[u], o);
            if (better(ov, oi, bv[u], bi[u])) {
                bv[u] = ov;
                bi[u] = oi;
            }
        }
    if (lane < 4) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            rv[warp][2 * lane + u] = bv[u];
            ri[warp][2 * lane + u] = bi[u];
        }
    }
    __syncthreads();
    if (tid < M) {
        float v = rv[0][tid];
        int32_t ix = ri[0][tid];
        for (int w = 1; w < kWarps; ++w)
            if (better(rv[w][tid], ri[w][tid], v, ix)) {
                v = rv[w][tid];
                ix = ri[w][tid];
            }
        p.part_val[blockIdx.x * kMaxM + tid] = v;
        p.part_idx[blockIdx.x * kMaxM + tid] = ix;
    }

    // 7. the last CTA to finish reduces every CTA's partial
    __syncthreads();
    if (tid == 0) {
        __threadfence();   // this CTA's partials before its count
        s_last = atomicAdd(p.done, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (!s_last)
        return;
    __threadfence();
    if (warp < M) {
        float v = -INFINITY;
        int32_t ix = 0x7FFFFFFF;
        for (int c = lane; c < (int)gridDim.x; c += 32) {
            const float ov = __ldcg(p.part_val + c * kMaxM + warp);
            const int32_t oi = __ldcg(p.part_idx + c * kMaxM + warp);
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
            s_arg[warp] = ix;
            p.argmax[warp] = ix;
            if (p.maxlogit)
                p.maxlogit[warp] = v;
        }
    }
    __syncthreads();
    if (tid == 0) {
        if (p.out)
            accept_greedy(s_arg, p.draft, M, p.out);
        *p.done = 0u;   // ready for the next launch on this workspace
    }
}

// CTAs for V rows: one per SM, fewer when there are not enough tiles.
inline int grid_for(int64_t V, int sms)
{
    const int64_t tiles = (V + kRows - 1) / kRows;
    const int64_t need = (tiles + kWarps - 1) / kWarps;
    const int64_t g = need < sms ? need : sms;
    return g < 1 ? 1 : static_cast<int>(g < kMaxParts ? g : kMaxParts);
}

}  // namespace fp8head
}  // namespace fgm
