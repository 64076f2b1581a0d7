// Shared definitions of the CUDA library: model constants, workspace layout,
// number-format helpers and small warp/block reductions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fgm.h"

namespace fgm {

constexpr int kH = FGM_HIDDEN;         // hidden width
constexpr int kF = FGM_FFN;            // expert FFN width
constexpr int kE = FGM_EXPERTS;        // routed experts
constexpr int kNE = kE + FGM_SHARED;   // experts stored per layer
constexpr int kK = FGM_TOPK;           // routed experts per token
constexpr int kMaxM = FGM_MAX_M;       // tokens per call
constexpr int kShared = kE;            // index of the shared expert
constexpr int kMaxSlots = kMaxM * kK + 1;  // distinct routed experts + shared
constexpr int kMaxDense = 3;               // 704-wide parts of a dense shared MLP (up to 2112 wide)
constexpr int kMaxSlotsAll = kMaxM * kK + kMaxDense;   // routed + dense parts (per-stage kernels)
constexpr int kMaxParts = 2048;        // lm_head per-CTA partials kept in the workspace
constexpr float kEps = FGM_RMS_EPS;
constexpr int kSyncLmHeadDone = 127;   // workspace sync word counting finished FP8 lm_head CTAs
constexpr int kSyncTileCount = 2;      // sync words [2, 98): down tiles taken per slot, by layer parity
constexpr int kSyncTileStride = 48;    // (the persistent kernel's tensor-memory down phase, M <= 5)
static_assert(kSyncTileCount + 2 * kSyncTileStride <= kSyncLmHeadDone, "sync words overlap");

// Device scratch carved out of the caller's workspace (see ws_layout()).
struct Ws {
    float *h;          // [8][2816] fp32 residual stream
    float *xn;         // [8][2816] fp32 layer input (normed in the stack)
    float *acc;        // [8][2816] fp32 layer output accumulator
    float *logits;     // [8][128] router logits (bias included)
    int32_t *meta;     // [0] = distinct routed experts U, [1 + s] = expert of slot s (slots U..: the
                       // shared expert, or the parts kE + p of a dense shared MLP)
    float *comb;       // [67][8] routing weight of slot s for token t (0 when not routed)
    float *act;        // [2][67][8][704] weighted gated activations per slot and token (the staged
                       // path uses buffer 0; the persistent kernel alternates by layer over 65 slots)
    int32_t *ids;      // [8][8] chosen experts of the last routed layer
    float *wts;        // [8][8] their weights
    float *part_val;   // [kMaxParts][8] lm_head per-CTA best logit
    int32_t *part_idx; // [kMaxParts][8] and its row
    uint16_t *hb;      // [8][2816] bf16 lm_head input of the verify step
    int32_t *argmax;   // [8]
    uint16_t *io_x;    // [8][2816] staging of host inputs
    int32_t *io_draft; // [8]
    int32_t *io_out;   // [2]
    int32_t *status;   // [1] FGM_STATUS_* bits
    unsigned *sync;    // [128] [0] grid barrier, [1] exit count, [kSyncTileCount + 48 parity + s] down
                       // tiles taken from slot s, [kSyncLmHeadDone] CTAs done in the FP8 lm_head
    uint8_t *xterms;   // [8][3][2816] E4M3 terms of the gate/up input of the current layer
    float *xscale;     // [8][11] their power-of-two scale per token and 256-wide K-slice
    float *part_sum;   // [kMaxParts][8] sampling: per-CTA sum of exp((z - part_val) / T)
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Byte offsets of every region; the same function serves host and device.
struct WsOffsets {
    size_t h, xn, acc, logits, meta, comb, act, ids, wts, part_val, part_idx, hb, argmax, io_x,
        io_draft, io_out, status, sync, xterms, xscale, part_sum, total;
};

inline WsOffsets ws_offsets()
{
    WsOffsets o;
    size_t p = 0;
    auto take = [&](size_t bytes) {
        size_t at = p;
        p = align_up(p + bytes, 256);
        return at;
    };
    o.h = take(sizeof(float) * kMaxM * kH);
    o.xn = take(sizeof(float) * kMaxM * kH);
    o.acc = take(sizeof(float) * kMaxM * kH);
    o.logits = take(sizeof(float) * kMaxM * kE);
    o.meta = take(sizeof(int32_t) * (kMaxSlotsAll + 8));
    o.comb = take(sizeof(float) * kMaxSlotsAll * kMaxM);
    o.act = take(sizeof(float) * 2 * kMaxSlotsAll * kMaxM * kF);
    o.ids = take(sizeof(int32_t) * kMaxM * kK);
    o.wts = take(sizeof(float) * kMaxM * kK);
    o.part_val = take(sizeof(float) * kMaxParts * kMaxM);
    o.part_idx = take(sizeof(int32_t) * kMaxParts * kMaxM);
    o.hb = take(sizeof(uint16_t) * kMaxM * kH);
    o.argmax = take(sizeof(int32_t) * kMaxM);
    o.io_x = take(sizeof(uint16_t) * kMaxM * kH);
    o.io_draft = take(sizeof(int32_t) * kMaxM);
    o.io_out = take(sizeof(int32_t) * 2);
    o.status = take(sizeof(int32_t) * 64);
    o.sync = take(sizeof(unsigned) * 128);
    o.xterms = take(static_cast<size_t>(kMaxM) * 3 * kH);
    o.xscale = take(sizeof(float) * kMaxM * 11);
    o.part_sum = take(sizeof(float) * kMaxParts * kMaxM);
    o.total = p;
    return o;
}

inline Ws ws_carve(void *base)
{
    WsOffsets o = ws_offsets();
    char *b = static_cast<char *>(base);
    Ws w;
    w.h = reinterpret_cast<float *>(b + o.h);
    w.xn = reinterpret_cast<float *>(b + o.xn);
    w.acc = reinterpret_cast<float *>(b + o.acc);
    w.logits = reinterpret_cast<float *>(b + o.logits);
    w.meta = reinterpret_cast<int32_t *>(b + o.meta);
    w.comb = reinterpret_cast<float *>(b + o.comb);
    w.act = reinterpret_cast<float *>(b + o.act);
    w.ids = reinterpret_cast<int32_t *>(b + o.ids);
    w.wts = reinterpret_cast<float *>(b + o.wts);
    w.part_val = reinterpret_cast<float *>(b + o.part_val);
    w.part_idx = reinterpret_cast<int32_t *>(b + o.part_idx);
    w.hb = reinterpret_cast<uint16_t *>(b + o.hb);
    w.argmax = reinterpret_cast<int32_t *>(b + o.argmax);
    w.io_x = reinterpret_cast<uint16_t *>(b + o.io_x);
    w.io_draft = reinterpret_cast<int32_t *>(b + o.io_draft);
    w.io_out = reinterpret_cast<int32_t *>(b + o.io_out);
    w.status = reinterpret_cast<int32_t *>(b + o.status);
    w.sync = reinterpret_cast<unsigned *>(b + o.sync);
    w.xterms = reinterpret_cast<uint8_t *>(b + o.xterms);
    w.xscale = reinterpret_cast<float *>(b + o.xscale);
    w.part_sum = reinterpret_cast<float *>(b + o.part_sum);
    return w;
}

// Optional dense shared MLP of the per-stage layer kernels, in its natural
// layout: gate/up [parts * 704][2816], down [2816][parts * 704] (row stride
// parts * 704), fp32 row scales. Part p acts as expert kE + p: gate/up rows
// p * 704 .. and down columns p * 704 .., with the down rows' full-width
// scales. parts = 0: the layer's own shared expert.
struct DenseArgs {
    const uint8_t *gq;
    const float *gs;
    const uint8_t *uq;
    const float *us;
    const uint8_t *dq;
    const float *ds;
    int parts;
};

// ---------------------------------------------------------------- formats

// Four E4M3 codes (byte i = element i) to fp32 through the hardware
// E4M3x2 -> f16x2 conversion; every E4M3 value is exact in f16 and f32.
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float *o)
{
    __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w & 0xFFFFu), __NV_E4M3);
    __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w >> 16), __NV_E4M3);
    float2 a = __half22float2(__half2(lo));
    float2 b = __half22float2(__half2(hi));
    o[0] = a.x;
    o[1] = a.y;
    o[2] = b.x;
    o[3] = b.y;
}

__device__ __forceinline__ void e4m3x16_to_f32(const uint4 &v, float *o)
{
    e4m3x4_to_f32(v.x, o);
    e4m3x4_to_f32(v.y, o + 4);
    e4m3x4_to_f32(v.z, o + 8);
    e4m3x4_to_f32(v.w, o + 12);
}

// Two bf16 (low half = element 0) to fp32: a bf16 is the top half of a binary32.
__device__ __forceinline__ float2 bf16x2_to_f32(uint32_t w)
{
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

__device__ __forceinline__ uint16_t f32_to_bf16(float f)
{
    __nv_bfloat16 b = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t *>(&b);
}

// tanh-approximated GELU: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))).
__device__ __forceinline__ float gelu_tanh(float x)
{
    const float k = 0.7978845608028654f;
    return 0.5f * x * (1.0f + tanhf(k * (x + 0.044715f * x * x * x)));
}

// Larger logit wins; equal logits go to the smaller index.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi)
{
    return v > bv || (v == bv && i < bi);
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

}  // namespace fgm
