// Straightforward kernels of the verify step: one launch per stage, CUDA-core
// fp32 arithmetic, 16-byte coalesced weight loads. They define the step's
// numerics for the library and serve the single-layer entry points; the fused
// persistent kernel in fused_step.cuh reuses the same stage order.
#pragma once

#include "common.cuh"

namespace fgm {

// ---------------------------------------------------------------- small stages

// xn[t] = float(x[t]) and acc[t] = 0 for the single-layer call.
__global__ void k_layer_prep(const uint16_t *__restrict__ x, int M, float *__restrict__ xn,
                             float *__restrict__ acc)
{
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < M * kH; i += gridDim.x * blockDim.x) {
        xn[i] = bf16_to_f32(x[i]);
        acc[i] = 0.0f;
    }
}

__global__ void k_bf16_to_f32(const uint16_t *__restrict__ x, int n, float *__restrict__ out)
{
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
        out[i] = bf16_to_f32(x[i]);
}

__global__ void k_f32_to_bf16(const float *__restrict__ x, int n, uint16_t *__restrict__ out)
{
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
        out[i] = f32_to_bf16(x[i]);
}

// Unit-gain RMSNorm of row blockIdx.x: xn = h / sqrt(mean(h^2) + eps); fp32
// and/or bf16 output.
__global__ void __launch_bounds__(256) k_rmsnorm(const float *__restrict__ h, float *__restrict__ xn,
                                                 uint16_t *__restrict__ xb)
{
    __shared__ float red[8];
    const int t = blockIdx.x;
    const float *row = h + (size_t)t * kH;
    float ss = 0.0f;
    for (int j = threadIdx.x; j < kH; j += blockDim.x)
        ss += row[j] * row[j];
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x < 32) {
        float v = threadIdx.x < 8 ? red[threadIdx.x] : 0.0f;
        v = warp_sum(v);
        if (threadIdx.x == 0)
            red[0] = v;
    }
    __syncthreads();
    const float r = 1.0f / sqrtf(red[0] / (float)kH + kEps);
    for (int j = threadIdx.x; j < kH; j += blockDim.x) {
        const float v = row[j] * r;
        if (xn)
            xn[(size_t)t * kH + j] = v;
        if (xb)
            xb[(size_t)t * kH + j] = f32_to_bf16(v);
    }
}

// Router logits, one CTA per expert e: logits[t][e] = W_r[e] . xn[t] + b[e].
__global__ void __launch_bounds__(256) k_router_logits(const float *__restrict__ xn, int M,
                                                       const uint16_t *__restrict__ wr,
                                                       const float *__restrict__ bias,
                                                       float *__restrict__ logits)
{
    __shared__ float red[8][kMaxM];
    const int e = blockIdx.x;
    float s[kMaxM];
#pragma unroll
    for (int t = 0; t < kMaxM; ++t)
        s[t] = 0.0f;
    for (int j = threadIdx.x; j < kH; j += blockDim.x) {
        const float w = bf16_to_f32(wr[(size_t)e * kH + j]);
#pragma unroll
        for (int t = 0; t < kMaxM; ++t)
            if (t < M)
                s[t] += w * xn[(size_t)t * kH + j];
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int t = 0; t < kMaxM; ++t) {
        const float v = warp_sum(s[t]);
        if (lane == 0)
            red[warp][t] = v;
    }
    __syncthreads();
    if (threadIdx.x < M) {
        float v = 0.0f;
        for (int w = 0; w < 8; ++w)
            v += red[w][threadIdx.x];
        logits[threadIdx.x * kE + e] = v + (bias ? bias[e] : 0.0f);
    }
}

// Softmax + top-8 + renormalisation of one token's 128 logits by one warp.
// Lane l holds logits l, l+32, l+64, l+96. Ties go to the lower index; NaN
// logits count as -inf and raise a status bit. Renormalised weights are
// exp(l_i - l_max) / sum over the chosen exp(l_j - l_max), which equals the
// softmax over all 128 divided by the chosen mass.
__device__ __forceinline__ void warp_topk8(const float *__restrict__ lrow, int lane, int32_t *ids,
                                           float *wts, int32_t *status)
{
    float v[4];
    bool bad = false;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        v[q] = lrow[lane + 32 * q];
        if (isnan(v[q])) {
            v[q] = -INFINITY;
            bad = true;
        }
    }
    if (__any_sync(0xFFFFFFFFu, bad) && lane == 0)
        atomicOr(status, FGM_STATUS_NONFINITE_LOGITS);
    unsigned taken = 0;
    float top_v[kK];
    int top_i[kK];
#pragma unroll
    for (int r = 0; r < kK; ++r) {
        float bv = -INFINITY;
        int bi = 0x7FFFFFFF;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int idx = lane + 32 * q;
            if (!(taken & (1u << q)) && better(v[q], idx, bv, bi)) {
                bv = v[q];
                bi = idx;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
            const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
            if (better(ov, oi, bv, bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if ((bi & 31) == lane)
            taken |= 1u << (bi >> 5);
        top_v[r] = bv;
        top_i[r] = bi;
    }
    float ex[kK], z = 0.0f;
#pragma unroll
    for (int r = 0; r < kK; ++r) {
        ex[r] = top_v[0] == -INFINITY ? 1.0f : expf(top_v[r] - top_v[0]);
        z += ex[r];
    }
    if (lane == 0) {
#pragma unroll
        for (int r = 0; r < kK; ++r) {
            ids[r] = top_i[r];
            wts[r] = ex[r] / z;
        }
    }
}

// Top-k for all tokens, then the distinct-expert list: slots 0..U-1 hold the
// distinct routed experts in ascending id order, slots U..U+n_shared-1 the
// shared part(s) (expert kE + p). comb[s][t] is token t's routing weight for
// slot s (0 if not routed, 1 for a shared slot), so every slot can be
// evaluated for all tokens and weighted afterwards.
__global__ void __launch_bounds__(256) k_topk_dedup(const float *__restrict__ logits, int M, int n_shared,
                                                    int32_t *__restrict__ meta,
                                                    float *__restrict__ comb,
                                                    int32_t *__restrict__ ids_out,
                                                    float *__restrict__ w_out,
                                                    int32_t *__restrict__ status)
{
    __shared__ int32_t s_ids[kMaxM][kK];
    __shared__ float s_w[kMaxM][kK];
    __shared__ int32_t mark[kE];
    __shared__ int32_t slot_of[kE];
    __shared__ int32_t s_nu;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < kE; i += blockDim.x)
        mark[i] = 0;
    if (warp < M)
        warp_topk8(logits + warp * kE, lane, s_ids[warp], s_w[warp], status);
    __syncthreads();
    if (threadIdx.x < M * kK)
        mark[s_ids[threadIdx.x / kK][threadIdx.x % kK]] = 1;
    __syncthreads();
    if (warp == 0) {
        int base = 0;
        for (int q = 0; q < kE / 32; ++q) {
            const int e = q * 32 + lane;
            const bool m = mark[e] != 0;
            const unsigned b = __ballot_sync(0xFFFFFFFFu, m);
            const int pos = base + __popc(b & ((1u << lane) - 1u));
            if (m) {
                meta[1 + pos] = e;
                slot_of[e] = pos;
            }
            base += __popc(b);
        }
        if (lane == 0) {
            meta[0] = base;
            for (int p = 0; p < n_shared; ++p)
                meta[1 + base + p] = kShared + p;
            s_nu = base;
        }
    }
    __syncthreads();
    const int n_slots = s_nu + n_shared;
    for (int i = threadIdx.x; i < n_slots * kMaxM; i += blockDim.x)
        comb[i] = 0.0f;
    __syncthreads();
    if (threadIdx.x < M * kK) {
        const int t = threadIdx.x / kK, r = threadIdx.x % kK;
        comb[slot_of[s_ids[t][r]] * kMaxM + t] = s_w[t][r];
        if (ids_out) {
            ids_out[t * kK + r] = s_ids[t][r];
            if (w_out)
                w_out[t * kK + r] = s_w[t][r];
        }
    }
    if (threadIdx.x < n_shared * kMaxM)
        comb[(s_nu + threadIdx.x / kMaxM) * kMaxM + threadIdx.x % kMaxM] = threadIdx.x % kMaxM < M ? 1.0f : 0.0f;
}

// ---------------------------------------------------------------- experts

// Gate/up + gated GELU. Grid (22, 67): blockIdx.y is the slot, each CTA covers
// 32 rows of the 704 (8 warps x 4 rows). A warp streams gate row i and up row
// i with 16-byte loads and keeps M dot products of each; the activation
// act[s][t][i] = comb[s][t] * gelu_tanh(s_g g) * (s_u u). Slots of expert
// kE + p read part p of the dense shared MLP when dn.parts > 0.
template <int M>
__global__ void __launch_bounds__(256) k_gateup_basic(const uint8_t *__restrict__ gq,
                                                      const float *__restrict__ gs,
                                                      const uint8_t *__restrict__ uq,
                                                      const float *__restrict__ us,
                                                      const float *__restrict__ xn,
                                                      const int32_t *__restrict__ meta,
                                                      const float *__restrict__ comb,
                                                      float *__restrict__ act, DenseArgs dn)
{
    extern __shared__ float4 smem4[];
    float *sx = reinterpret_cast<float *>(smem4);
    const int slot = blockIdx.y;
    if (slot >= meta[0] + (dn.parts ? dn.parts : 1))
        return;
    int expert = meta[1 + slot];
    if (expert >= kE && dn.parts) {   // part p of the dense MLP: the same layout as an expert
        gq = dn.gq;
        gs = dn.gs;
        uq = dn.uq;
        us = dn.us;
        expert -= kE;
    }
    for (int i = threadIdx.x; i < M * kH / 4; i += blockDim.x)
        smem4[i] = reinterpret_cast<const float4 *>(xn)[i];
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int r = 0; r < 4; ++r) {
        const int row = (blockIdx.x * 8 + warp) * 4 + r;
        if (row >= kF)
            break;
        const uint8_t *grow = gq + ((size_t)expert * kF + row) * kH;
        const uint8_t *urow = uq + ((size_t)expert * kF + row) * kH;
        float ag[M], au[M];
#pragma unroll
        for (int t = 0; t < M; ++t)
            ag[t] = au[t] = 0.0f;
#pragma unroll
        for (int c = 0; c < 6; ++c) {
            const int o = c * 512 + lane * 16;
            if (o < kH) {
                const uint4 g4 = __ldg(reinterpret_cast<const uint4 *>(grow + o));
                const uint4 u4 = __ldg(reinterpret_cast<const uint4 *>(urow + o));
                float wg[16], wu[16];
                e4m3x16_to_f32(g4, wg);
                e4m3x16_to_f32(u4, wu);
#pragma unroll
                for (int t = 0; t < M; ++t) {
                    const float *xp = sx + t * kH + o;
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        ag[t] += wg[i] * xp[i];
                        au[t] += wu[i] * xp[i];
                    }
                }
            }
        }
#pragma unroll
        for (int t = 0; t < M; ++t) {
            ag[t] = warp_sum(ag[t]);
            au[t] = warp_sum(au[t]);
        }
        if (lane == 0) {
            const float sg = gs[(size_t)expert * kF + row], su = us[(size_t)expert * kF + row];
#pragma unroll
            for (int t = 0; t < M; ++t)
                act[((size_t)slot * kMaxM + t) * kF + row] =
                    comb[slot * kMaxM + t] * gelu_tanh(sg * ag[t]) * (su * au[t]);
        }
    }
}

// Down projection + combine. Grid (88, 67): slot blockIdx.y, 32 output rows per
// CTA (8 warps x 4 rows). out[t][j] += s_d[j] * (Q_d[j] . act[s][t]); several
// slots add into the same output element with fp32 atomics. Part p of a dense
// shared MLP reads columns p * 704 .. of its full-width down rows and their
// scales.
template <int M>
__global__ void __launch_bounds__(256) k_down_basic(const uint8_t *__restrict__ dq,
                                                    const float *__restrict__ ds,
                                                    const float *__restrict__ act,
                                                    const int32_t *__restrict__ meta,
                                                    float *__restrict__ out, DenseArgs dn)
{
    __shared__ __align__(16) float sa[M * kF];
    const int slot = blockIdx.y;
    if (slot >= meta[0] + (dn.parts ? dn.parts : 1))
        return;
    const int expert = meta[1 + slot];
    const bool dense = expert >= kE && dn.parts;
    // row j of this slot's down matrix and its scale
    const size_t row_stride = dense ? (size_t)dn.parts * kF : kF;
    const uint8_t *dbase = dense ? dn.dq + (size_t)(expert - kE) * kF : dq + (size_t)expert * kH * kF;
    const float *sbase = dense ? dn.ds : ds + (size_t)expert * kH;
    for (int i = threadIdx.x; i < M * kF; i += blockDim.x)
        sa[i] = act[((size_t)slot * kMaxM + i / kF) * kF + i % kF];
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int r = 0; r < 4; ++r) {
        const int j = (blockIdx.x * 8 + warp) * 4 + r;
        if (j >= kH)
            break;
        const uint8_t *drow = dbase + (size_t)j * row_stride;
        float a[M];
#pragma unroll
        for (int t = 0; t < M; ++t)
            a[t] = 0.0f;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int o = c * 512 + lane * 16;
            if (o < kF) {
                const uint4 d4 = __ldg(reinterpret_cast<const uint4 *>(drow + o));
                float wd[16];
                e4m3x16_to_f32(d4, wd);
#pragma unroll
                for (int t = 0; t < M; ++t) {
                    const float *ap = sa + t * kF + o;
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        a[t] += wd[i] * ap[i];
                }
            }
        }
#pragma unroll
        for (int t = 0; t < M; ++t)
            a[t] = warp_sum(a[t]);
        if (lane == 0) {
            const float sd = sbase[j];
#pragma unroll
            for (int t = 0; t < M; ++t)
                atomicAdd(out + (size_t)t * kH + j, sd * a[t]);
        }
    }
}

// ---------------------------------------------------------------- lm_head

// lm_head + per-CTA argmax. Warps stride over vocabulary rows; each row is
// 5632 bytes = 11 16-byte loads per lane. Rows are visited in increasing
// order per warp, so a strict comparison keeps the lowest index on ties.
template <int M>
__global__ void __launch_bounds__(256) k_lmhead_basic(const uint16_t *__restrict__ emb, int64_t V,
                                                      const uint16_t *__restrict__ hb,
                                                      float *__restrict__ part_val,
                                                      int32_t *__restrict__ part_idx)
{
    extern __shared__ float4 smem4[];
    float *sh = reinterpret_cast<float *>(smem4);
    __shared__ float rv[8][kMaxM];
    __shared__ int32_t ri[8][kMaxM];
    for (int i = threadIdx.x; i < M * kH; i += blockDim.x)
        sh[i] = bf16_to_f32(hb[i]);
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float best[M];
    int32_t bidx[M];
#pragma unroll
    for (int t = 0; t < M; ++t) {
        best[t] = -INFINITY;
        bidx[t] = 0x7FFFFFFF;
    }
    for (int64_t row = (int64_t)blockIdx.x * 8 + warp; row < V; row += (int64_t)gridDim.x * 8) {
        const uint16_t *er = emb + row * kH;
        float s[M];
#pragma unroll
        for (int t = 0; t < M; ++t)
            s[t] = 0.0f;
#pragma unroll
        for (int c = 0; c < 11; ++c) {
            const int o = c * 256 + lane * 8;
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(er + o));
            float w[8];
            float2 p;
            p = bf16x2_to_f32(v.x); w[0] = p.x; w[1] = p.y;
            p = bf16x2_to_f32(v.y); w[2] = p.x; w[3] = p.y;
            p = bf16x2_to_f32(v.z); w[4] = p.x; w[5] = p.y;
            p = bf16x2_to_f32(v.w); w[6] = p.x; w[7] = p.y;
#pragma unroll
            for (int t = 0; t < M; ++t) {
                const float *xp = sh + t * kH + o;
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    s[t] += w[i] * xp[i];
            }
        }
#pragma unroll
        for (int t = 0; t < M; ++t) {
            const float z = warp_sum(s[t]);
            if (z > best[t]) {
                best[t] = z;
                bidx[t] = (int32_t)row;
            }
        }
    }
    if (lane == 0) {
#pragma unroll
        for (int t = 0; t < M; ++t) {
            rv[warp][t] = best[t];
            ri[warp][t] = bidx[t];
        }
    }
    __syncthreads();
    if (threadIdx.x < M) {
        const int t = threadIdx.x;
        float bv = rv[0][t];
        int32_t bi = ri[0][t];
        for (int w = 1; w < 8; ++w)
            if (better(rv[w][t], ri[w][t], bv, bi)) {
                bv = rv[w][t];
                bi = ri[w][t];
            }
        part_val[blockIdx.x * kMaxM + t] = bv;
        part_idx[blockIdx.x * kMaxM + t] = bi;
    }
}

// Greedy acceptance on tokens already in shared or global memory.
__device__ __forceinline__ void accept_greedy(const int32_t *target, const int32_t *draft, int M,
                                              int32_t *out)
{
    int a = 0;
    while (a < M - 1 && draft[a] == target[a])
        ++a;
    out[0] = a;
    out[1] = target[a];
}

// Cross-CTA argmax (one warp per token) and, if `out` is given, greedy acceptance.
__global__ void __launch_bounds__(256) k_argmax_final(const float *__restrict__ part_val,
                                                      const int32_t *__restrict__ part_idx, int G,
                                                      int M, int32_t *__restrict__ argmax,
                                                      float *__restrict__ maxlogit,
                                                      const int32_t *__restrict__ draft,
                                                      int32_t *__restrict__ out,
                                                      int32_t *__restrict__ status)
{
    __shared__ int32_t s_arg[kMaxM];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp < M) {
        float bv = -INFINITY;
        int32_t bi = 0x7FFFFFFF;
        for (int g = lane; g < G; g += 32) {
            const float v = part_val[g * kMaxM + warp];
            const int32_t i = part_idx[g * kMaxM + warp];
            if (better(v, i, bv, bi)) {
                bv = v;
                bi = i;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
            const int32_t oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
            if (better(ov, oi, bv, bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if (lane == 0) {
            if (bi == 0x7FFFFFFF) {  // every logit was NaN
                bi = 0;
                atomicOr(status, FGM_STATUS_NONFINITE_LOGITS);
            }
            s_arg[warp] = bi;
            if (argmax)
                argmax[warp] = bi;
            if (maxlogit)
                maxlogit[warp] = bv;
        }
    }
    __syncthreads();
    if (out && threadIdx.x == 0)
        accept_greedy(s_arg, draft, M, out);
}

__global__ void k_spec_verify(const int32_t *__restrict__ target, const int32_t *__restrict__ draft,
                              int M, int32_t *__restrict__ out)
{
    if (threadIdx.x == 0 && blockIdx.x == 0)
        accept_greedy(target, draft, M, out);
}

}  // namespace fgm
