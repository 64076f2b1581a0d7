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
//  * One CTA per SM, 16 warps. Warp w owns whole 16-row tiles of the
//    vocabulary, tiles w, w + W, ... (W = warps in the grid), and reads each
//    tile's 45 KB once with 16-byte streaming loads that skip L1. A lane reads
//    16 bytes of row g = lane / 4 and of row g + 8 per 64-byte K-block, so four
//    lanes cover 64 contiguous bytes of a row and a warp step touches full
//    32-byte sectors only.
//  * Products on the tensor cores: mma.sync m16n8k16 with f16 operands and
//    fp32 accumulation. The E4M3 codes become f16 through the hardware
//    conversion (every E4M3 value is exact in f16); the 8 MMA columns are the
//    tokens (absent tokens are zero). Within a K-block the lane's 16 bytes are
//    four k16 slices: slice i takes bytes 4i..4i+3, the A fragment's k pairs
//    (2t, 2t+1) and (2t+8, 2t+9) being bytes (4i, 4i+1) and (4i+2, 4i+3) of
//    lane t's chunk. The B fragment maps k the same way (it depends on t only),
//    so every product meets its own hidden element.
//  * The hidden rows live in shared memory as f16, each token scaled by a
//    power of two 2^s so that its largest |h| lies in [2^14, 2^15): bf16
//    inputs of any magnitude fit f16's range, the scaling is exact, and the
//    logit is unscaled exactly by 2^-s in the epilogue.
//  * Loads run one pipeline step (4 K-blocks, 4 KB per warp) ahead of the
//    products, including across tile boundaries, so ~64 KB per SM is in flight.
//  * Epilogue per tile: row scale, unscale, running (max, lowest index) per
//    token; then a warp and CTA reduction to one partial per CTA, reduced
//    across CTAs by k_argmax_final.
#pragma once

#include "common.cuh"

namespace fgm {
namespace fp8head {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kRows = 16;                  // vocabulary rows per warp tile (the MMA's M)
constexpr int kPitch = kH + 8;             // f16 per token row in shared memory (16-byte pad)
constexpr int kBlock = 64;                 // K elements per lane quad and K-block (4 lanes x 16 bytes)
constexpr int kBlocks = kH / kBlock;       // 44 K-blocks per row
constexpr int kGroup = 4;                  // K-blocks per pipeline step
constexpr int kSteps = kBlocks / kGroup;   // 11 steps per tile
static_assert(kH % (kBlock * kGroup) == 0, "hidden width must split into whole pipeline steps");

// 16 bytes of a stream read once: no L1 allocation, L2 fetches 256-byte spans.
__device__ __forceinline__ uint4 ld_stream16(const uint8_t *p)
{
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

// Two E4M3 codes (low byte = lower k) to an f16x2 word (low half = lower k); exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two)
{
    const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two & 0xFFFFu), __NV_E4M3);
    return static_cast<uint32_t>(r.x) | (static_cast<uint32_t>(r.y) << 16);
}

__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Per-CTA argmax partials over the rows this CTA's warps visit:
// part_val/part_idx[blockIdx.x][t] for t < M (ties to the lower row).
__global__ void __launch_bounds__(kThreads, 1)
    k_lmhead_fp8(const uint8_t *__restrict__ q, const float *__restrict__ scale, int V,
                 const uint16_t *__restrict__ hb, int M, float *__restrict__ part_val,
                 int32_t *__restrict__ part_idx)
{
    __shared__ __align__(16) uint16_t hs[kMaxM * kPitch];   // f16 bits of h * 2^s, zero rows for t >= M
    __shared__ unsigned amax_bits[kMaxM];
    __shared__ float up[kMaxM], down[kMaxM];                 // 2^s and 2^-s per token
    __shared__ float rv[kWarps][kMaxM];
    __shared__ int32_t ri[kWarps][kMaxM];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;

    // 1. largest finite |h| per token (non-negative floats order like their bits)
    for (int tk = warp; tk < kMaxM; tk += kWarps) {
        unsigned m = 0;
        if (tk < M)
            for (int k = lane; k < kH; k += 32) {
                const float a = fabsf(bf16_to_f32(hb[(size_t)tk * kH + k]));
                if (a < INFINITY)
                    m = max(m, __float_as_uint(a));
            }
        m = __reduce_max_sync(0xFFFFFFFFu, m);
        if (lane == 0)
            amax_bits[tk] = m;
    }
    __syncthreads();
    // 2. s = 141 - biased exponent of that max puts it in [2^14, 2^15); a zero or
    //    subnormal max keeps s = 0. For finite bf16 maxima s >= -113; s <= 126
    //    keeps 2^s and 2^-s normal floats
    if (tid < kMaxM) {
        const int ef = static_cast<int>(amax_bits[tid] >> 23);
        int s = ef == 0 ? 0 : 141 - ef;
        s = min(126, s);
        up[tid] = __uint_as_float(static_cast<unsigned>(127 + s) << 23);
        down[tid] = __uint_as_float(static_cast<unsigned>(127 - s) << 23);
    }
    __syncthreads();
    // 3. h * 2^s to f16 in shared memory
    for (int i = tid; i < kMaxM * (kH / 2); i += kThreads) {
        const int tk = i / (kH / 2), k2 = i - tk * (kH / 2);
        uint32_t w = 0;
        if (tk < M) {
            const float2 v = bf16x2_to_f32(*reinterpret_cast<const uint32_t *>(hb + (size_t)tk * kH + 2 * k2));
            const __half2 hv = __floats2half2_rn(v.x * up[tk], v.y * up[tk]);
            w = *reinterpret_cast<const uint32_t *>(&hv);
        }
        *reinterpret_cast<uint32_t *>(hs + tk * kPitch + 2 * k2) = w;
    }
    __syncthreads();

    // 4. stream the tiles
    const int T = (V + kRows - 1) / kRows;
    const int W = gridDim.x * kWarps;
    const uint16_t *hrow = hs + g * kPitch + 16 * t;   // B operand: token g, this lane's 16 k per block
    float bv[2] = {-INFINITY, -INFINITY};               // tokens 2t, 2t + 1
    int32_t bi[2] = {0x7FFFFFFF, 0x7FFFFFFF};

    // rows g and g + 8 of tile tl (rows past the end read row V - 1 and are dropped)
    auto row_ptrs = [&](int tl, const uint8_t *&pa, const uint8_t *&pb) {
        const int r0 = min(tl * kRows + g, V - 1), r1 = min(tl * kRows + g + 8, V - 1);
        pa = q + (size_t)r0 * kH + 16 * t;
        pb = q + (size_t)r1 * kH + 16 * t;
    };

    int tile = blockIdx.x * kWarps + warp;
    uint4 cur[kGroup][2], nxt[kGroup][2];
    const uint8_t *pa = q, *pb = q;
    if (tile < T) {
        row_ptrs(tile, pa, pb);
#pragma unroll
        for (int b = 0; b < kGroup; ++b) {
            cur[b][0] = ld_stream16(pa + b * kBlock);
            cur[b][1] = ld_stream16(pb + b * kBlock);
        }
    }
    while (tile < T) {
        const int ntile = tile + W;
        const uint8_t *na = pa, *nb = pb;
        if (ntile < T)
            row_ptrs(ntile, na, nb);
        const int r0 = tile * kRows + g, r1 = r0 + 8;
        const float s0 = scale[min(r0, V - 1)], s1 = scale[min(r1, V - 1)];
        float c[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int s = 0; s < kSteps; ++s) {
            if (s + 1 < kSteps) {
#pragma unroll
                for (int b = 0; b < kGroup; ++b) {
                    nxt[b][0] = ld_stream16(pa + ((s + 1) * kGroup + b) * kBlock);
                    nxt[b][1] = ld_stream16(pb + ((s + 1) * kGroup + b) * kBlock);
                }
            } else if (ntile < T) {
#pragma unroll
                for (int b = 0; b < kGroup; ++b) {
                    nxt[b][0] = ld_stream16(na + b * kBlock);
                    nxt[b][1] = ld_stream16(nb + b * kBlock);
                }
            }
#pragma unroll
            for (int b = 0; b < kGroup; ++b) {
                const int kb = s * kGroup + b;
                const uint4 h0 = *reinterpret_cast<const uint4 *>(hrow + kb * kBlock);
                const uint4 h1 = *reinterpret_cast<const uint4 *>(hrow + kb * kBlock + 8);
                const uint32_t hw[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
                const uint32_t wa[4] = {cur[b][0].x, cur[b][0].y, cur[b][0].z, cur[b][0].w};
                const uint32_t wb[4] = {cur[b][1].x, cur[b][1].y, cur[b][1].z, cur[b][1].w};
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    mma_f16(c, e4m3x2_to_f16x2(wa[i]), e4m3x2_to_f16x2(wb[i]), e4m3x2_to_f16x2(wa[i] >> 16),
                            e4m3x2_to_f16x2(wb[i] >> 16), hw[2 * i], hw[2 * i + 1]);
            }
#pragma unroll
            for (int b = 0; b < kGroup; ++b) {
                cur[b][0] = nxt[b][0];
                cur[b][1] = nxt[b][1];
            }
        }
        // c[u]: row r0, token 2t + u; c[2 + u]: row r1, token 2t + u
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int tk = 2 * t + u;
            if (tk < M) {
                const float dn = down[tk];
                if (r0 < V) {
                    const float z = c[u] * s0 * dn;
                    if (better(z, r0, bv[u], bi[u])) {
                        bv[u] = z;
                        bi[u] = r0;
                    }
                }
                if (r1 < V) {
                    const float z = c[2 + u] * s1 * dn;
                    if (better(z, r1, bv[u], bi[u])) {
                        bv[u] = z;
                        bi[u] = r1;
                    }
                }
            }
        }
        tile = ntile;
        pa = na;
        pb = nb;
    }

    // 5. warp (lanes of equal t), then CTA
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
        part_val[blockIdx.x * kMaxM + tid] = v;
        part_idx[blockIdx.x * kMaxM + tid] = ix;
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
