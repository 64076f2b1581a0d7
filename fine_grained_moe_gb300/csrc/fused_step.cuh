// Persistent verify-step kernel: one cooperative launch runs every layer of
// the MoE stack (and, for the verify step, the lm_head argmax and greedy
// accept).
//
// CTA layout: one CTA per SM; 11 MMA warps and 1 producer warp.
//  * The producer warp streams weight rows from HBM into a 4-slot shared
//    memory ring with cp.async.bulk (TMA bulk copies) completing on mbarriers.
//    Weight loads never depend on activations, so the producer runs ahead of
//    the consumers across phase boundaries; it only waits for the routing of
//    a layer before fetching that layer's routed experts.
//  * MMA warps split K: warp w owns a fixed 256-byte (gate/up, lm_head) or
//    64-byte (down) slice of every row and keeps the activations of that
//    slice in registers as mma B fragments. Each weight tile is 16 rows; the
//    products run on the tensor cores (mma.sync m16n8k32 E4M3 for experts,
//    m16n8k16 bf16 for the lm_head). The 11 partials of a tile meet in a
//    double-buffered shared-memory exchange; after one barrier, rotating
//    reducer warps sum them and apply the epilogue (row scales, gated GELU
//    and router weight for gate/up; row scales and fp32 atomic accumulation
//    into the residual for down; a running argmax per token for the lm_head).
//  * Experts read E4M3 weights as they are stored; the fp32 activations are
//    written as a sum of 3 E4M3 terms (each the rounding residual of the
//    previous one times 16) under a power-of-two scale per K-slice and token,
//    so products are exact and each activation carries <= 2^-12 relative
//    error. The B fragment columns hold (token, term) pairs: NB = 2 blocks of
//    8 columns for M <= 5, NB = 3 for M <= 8 (see column_of).
//
// Phases of layer l (every CTA):
//  A  RMSNorm sums of h and router logit e (CTA e < 128); the gate/up
//     activation terms are split once per grid (one warp per token and
//     K-slice) into the workspace.
//  -- grid barrier
//  B  softmax/top-8/renormalise + distinct-expert list (every CTA, same
//     result); gate/up tiles: shared-expert tiles, then routed ones, in whole
//     8-row tiles dealt over the CTAs.
//  C  down rows of every distinct expert and the shared one, dealt against
//     each CTA's gate/up tiles; each CTA polls the activation entries it
//     reads until their pending marker is gone (no barrier between B and C);
//     results (already weighted by the router) are added into the fp32
//     residual h with atomics.
//  -- grid barrier
// Verify step: final RMSNorm -> bf16, lm_head rows split over CTAs with a
// running argmax per token, then the last CTA to finish reduces the per-CTA
// winners and applies the greedy accept rule (no waiting involved).
#pragma once

#include <cuda.h>

#include <type_traits>

#include "common.cuh"

namespace fgm {
namespace fused {

constexpr int kMW = 11;                       // MMA warps (K-slices)
constexpr int kProdWarp = kMW;                // producer warp index
constexpr int kConsumers = kMW * 32;          // 352
constexpr int kThreads = kConsumers + 32;     // 384
constexpr int kStages = 4;                    // ring slots
constexpr int kRowStride = 2880;              // smem stride of a 2816-byte row (conflict-free 16-byte reads)
constexpr int kSlotBytes = 16 * kRowStride;   // 46080
constexpr int kDownTiles = 4;                 // 16-row down tiles per ring slot (64 x 704 bytes)
constexpr int kRouterCtas = 64;               // the last 64 CTAs compute the router logits,
constexpr int kRouterRows = FGM_EXPERTS / kRouterCtas;   // 2 rows each (fewer CTAs read the residual)
constexpr int kTerms = 3;                     // E4M3 terms per activation
constexpr int kSharedSlot = kMaxM * kK;     // first always-on slot: the shared expert, or dense part p at + p
constexpr uint32_t kActPending = 0x7FC0DEADu;   // NaN marker: activation row not written yet
constexpr int kMinCtas = 128;                 // the persistent kernel needs at least this many SMs
constexpr int kMaxGuRows = 8 * ((kMaxSlotsAll * (kF / 8) + kMinCtas - 1) / kMinCtas);   // routed row pairs per CTA
constexpr int kMaxDownRows = 16 * (kMaxSlotsAll * (kH / 16) / kMinCtas + 5);   // down rows per CTA (see down_rows)
constexpr int kMaxShTiles = (kMaxDense * (kF / 8) + kMinCtas - 1) / kMinCtas;   // always-on gate/up tiles per CTA

enum Mode { kModeLayer = 0, kModeStack = 1, kModeVerify = 2, kModeLmHead = 3 };
enum TileKind { kTileGateUp = 0, kTileDown = 1, kTileLmHead = 2 };

// Compile-time tile kind: each exchange site carries only its own epilogue.
template <int K>
struct KindTag {
    static constexpr int value = K;
};

struct Params {
    fgm_layer layers[FGM_MAX_LAYERS];
    int n_layers;
    int M;
    int mode;
    const uint16_t *x;      // bf16 [M][2816] input (lm_head mode: the hidden states)
    uint16_t *y;            // bf16 [M][2816] output (layer / stack)
    const uint16_t *emb;    // bf16 [V][2816] (verify, lm_head)
    int64_t V;
    const int32_t *draft;   // [M-1] (verify)
    int32_t *argmax;        // [M] (verify, lm_head)
    float *maxlogit;        // [M] (lm_head, optional)
    int32_t *out;           // [2] (verify)
    float *z;               // sampling at T > 0 (verify, lm_head): logits out [M][V]; null = greedy
    float inv_t;            // sampling: 1 / T
    const float *u_acc;     // sampling: [M-1] acceptance uniforms
    const float *u_next;    // sampling: [M] uniforms of the emitted sample
    int32_t *ids;           // layer: [M][8]; stack/verify: [L][M][8] trace; optional
    float *wts;             // layer: [M][8]; optional
    DenseArgs dense[FGM_MAX_LAYERS];   // NS = 3: each layer's always-on dense MLP (its 3 parts)
    int dense_parts;                   // 3 when the layers carry dense MLPs (NS = 3), else 0
    // tensor-memory down phase: each layer's down_q as [129 * 2816 rows][704 bytes],
    // 128 x 128-byte boxes in the 128-byte swizzle
    CUtensorMap dmap[FGM_MAX_LAYERS];
    Ws ws;
    long long timeout_ns;
    long long *trace;       // optional: %globaltimer stamps (see kTracePoints)
    int debug_stall;        // test hook: 1 + the layer that adds one grid barrier that can never
                            // complete (0: none)
};

// The dense variant's parameters (NS = 3): each layer's dense down matrix as
// [2816 rows][3 * 704 bytes] for the tensor-memory down phase, the same boxes
// (a part's tile starts at byte 704 p of its rows). A type of its own keeps
// the other instantiations' parameter block as small as it was.
struct ParamsDense : Params {
    CUtensorMap dmap_dense[FGM_MAX_LAYERS];
};

template <int NS>
using ParamsFor = typename std::conditional<(NS > 1), ParamsDense, Params>::type;

// Profiling aid (Params::trace): per layer kTracePoints phase stamps for every
// CTA, [(l * kTracePoints + k) * G + cta], then two end stamps per CTA, then
// for CTA G/2 only a per-stage timeline [l][kTraceStages][8] of SM clock64
// values = {producer issue, data landed, products done, slot released, last
// exchange posted, consumer wait begun, -, layer start}.
constexpr int kTracePoints = 12;
constexpr int kTraceStages = 48;
constexpr int kTraceDetail = 8;

struct __align__(128) Smem {
    uint8_t ring[kStages][kSlotBytes];
    float4 red[2][kMW][2][32];   // per-warp K-slice partials of up to 2 tiles, double-buffered
    float part[kMW][8];
    float part2[kRouterRows][kMW][8];
    float best_v[kMW][8];       // lm_head winners per reducing warp and token
    int32_t best_i[kMW][8];
    float samp_s[kMW][8];       // sampling: sum of exp((z - best_v) / T) per reducing warp and token
    float comb[2][kMaxSlotsAll][8];
    int32_t experts[2][kMaxSlotsAll];
    int32_t n_unique[2];
    int32_t tk_ids[8][8];
    float tk_w[8][8];
    int32_t mark[kE];
    int32_t slot_of[kE];
    float sc_g[kMaxGuRows + 8 * kMaxShTiles];   // gate/up row scales of this CTA's routed rows, then
    float sc_u[kMaxGuRows + 8 * kMaxShTiles];   // (from kMaxGuRows) its always-on rows
    alignas(16) float sc_d[kMaxDownRows];   // down row scales of this CTA's down rows of the layer
                                            // (tensor-memory phase: of its last kTcInfo tiles)
    int2 tinfo[8];              // tensor-memory down phase: (first row in the flattened (slot, row)
                                // space or -1 at the end, home slot 0/1) of tile sequence number % 8
    unsigned long long full[kStages];
    unsigned long long empty[kStages];
    unsigned long long route;
    unsigned long long tfull[2], tempty[2];   // tensor-memory down phase: accumulators full / read
    unsigned long long bready;                // tensor-memory down phase: second home slot's operand built
    unsigned long long mdone;                 // tensor-memory down phase: every product issued done
    uint32_t tmem_base;
    uint32_t tc_stage, tc_next;   // tensor-memory down phase: ring stages and tile numbers after it
    float dscale[2][8];         // tensor-memory down phase: activation-term scale per (slot, token)
    float tc_amax[8][2];        // tensor-memory down phase: half-row maxima of the first slot per token
    int abort;
    int last;
};

// ---------------------------------------------------------------- primitives

__device__ __forceinline__ uint32_t su32(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ long long gtime()
{
    long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(unsigned long long *b, int count)
{
    asm volatile("mbarrier.init.shared.b64 [%0], %1;" ::"r"(su32(b)), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(unsigned long long *b, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(unsigned long long *b)
{
    asm volatile("mbarrier.arrive.shared.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}

__device__ __forceinline__ bool mbar_try(unsigned long long *b, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(su32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait: gives up when the CTA's abort flag is raised or the kernel's
// deadline passes (then raises the abort flag and the status bit).
// On timeout the first wait to give up records where: status[1] = site, status[2] =
// block, status[3] = warp, status[4] = the stage/post index it waited for.
__device__ __noinline__ bool mbar_wait_slow(unsigned long long *b, uint32_t parity, Smem &s, long long deadline,
                                            int32_t *status, int site, int index)
{
    for (int it = 0;; ++it) {
        if (mbar_try(b, parity))
            return true;
        if ((it & 15) == 15) {
            if (*reinterpret_cast<volatile int *>(&s.abort))
                return false;
            if (gtime() > deadline) {
                *reinterpret_cast<volatile int *>(&s.abort) = 1;
                if (atomicOr(status, FGM_STATUS_WAIT_TIMEOUT) == 0) {
                    status[1] = site;
                    status[2] = blockIdx.x;
                    status[3] = threadIdx.x >> 5;
                    status[4] = index;
                }
                return false;
            }
        }
    }
}

// The common case inline (the phase has usually completed), the bounded
// slow path out of line: one copy of it keeps the kernel's hot loops small.
__device__ __forceinline__ bool mbar_wait(unsigned long long *b, uint32_t parity, Smem &s, long long deadline,
                                          int32_t *status, int site = 0, int index = 0)
{
#pragma unroll 1
    for (int it = 0; it < 8; ++it)
        if (mbar_try(b, parity))
            return true;
    return mbar_wait_slow(b, parity, s, deadline, status, site, index);
}

// 16-byte shared-memory load as volatile asm: it keeps its place ahead of the
// (volatile) mma instructions that consume it, so all of a stage's loads are
// in flight before the first product instead of one chunk at a time.
__device__ __forceinline__ uint4 lds128(const void *p)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))));
    return v;
}

// Starts an asynchronous HBM -> L2 copy (no completion tracking).
__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, unsigned long long *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(su32(dst)),
        "l"(src), "r"(bytes), "r"(su32(bar))
        : "memory");
}

// L2 policy for data read once per step (the weight streams): evicted first,
// so that the small data the layers re-read (activations, the residual, the
// next layer's router rows) stays in L2.
__device__ __forceinline__ uint64_t l2_evict_first()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void bulk_g2s_stream(void *dst, const void *src, uint32_t bytes, unsigned long long *bar,
                                                uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            su32(dst)),
        "l"(src), "r"(bytes), "r"(su32(bar)), "l"(pol)
        : "memory");
}

// ---------------------------------------------------------------- tcgen05
// The tensor-memory down phase (TCD): weights by TMA tensor copies into the
// ring, activations as E4M3 terms in shared memory, full-K accumulators in
// tensor memory, products by tcgen05.mma issued from one thread.
constexpr int kTcRows = 128;                 // rows per down tile (the MMA's M)
constexpr int kTcN = 16;                     // MMA N: 5 tokens x 3 terms (+ 1 zero column)
constexpr int kTcStagesPerTile = 3;          // K 0..255, 256..511, 512..767 (zeros past 704)
constexpr int kTcBoxBytes = kTcRows * 128;   // one 128-row x 128-byte box
constexpr int kTcBBytes = (kF / 16) * 256;   // B operand of one slot: 44 K-columns x 16 rows x 16 bytes
constexpr uint32_t kTcTmemCols = 32;         // two 16-column accumulators
constexpr int kTcInfo = 8;                   // tile records in flight (producer at most 4 tiles ahead of the epilogue)
static_assert(kTcInfo * kTcRows <= kMaxDownRows, "tile scales do not fit");
static_assert(5 * kK + 3 <= kSyncTileStride, "down-tile counters: slots at M <= 5 (up to three always-on parts)");
// instruction descriptor, kind::f8f6f4: D fp32, A and B E4M3, both K-major, N >> 3, M >> 4
constexpr uint32_t kTcIdesc = (1u << 4) | (static_cast<uint32_t>(kTcN >> 3) << 17) |
                              (static_cast<uint32_t>(kTcRows >> 4) << 24);

// A operand: K-major, 128-byte swizzle (8-row x 128-byte atoms 1024 bytes apart).
__device__ __forceinline__ uint64_t tc_desc_sw128(uint32_t addr)
{
    return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) | (1ull << 16) | (64ull << 32) | (1ull << 46) | (2ull << 61);
}

// B operand: K-major, no swizzle: core matrices of 8 rows x 16 bytes, 256 bytes
// apart along K (leading byte offset) and 128 bytes apart along N (stride byte offset).
__device__ __forceinline__ uint64_t tc_desc_nosw(uint32_t addr)
{
    return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) | (16ull << 16) | (8ull << 32) | (1ull << 46);
}

// Byte offset of (column n, k) in a B operand (see tc_desc_nosw).
__device__ __forceinline__ int tc_b_offset(int n, int k) { return (k >> 4) * 256 + (n >> 3) * 128 + (n & 7) * 16 + (k & 15); }

__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(kTcIdesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_commit(unsigned long long *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

// 16 consecutive fp32 columns of this thread's lane
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i)
        v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap *map, int x, int y, unsigned long long *bar,
                                       uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3}], "
        "[%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(su32(bar)), "l"(pol)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_n(unsigned long long *b, uint32_t n)
{
    asm volatile("mbarrier.arrive.shared.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(n) : "memory");
}

// Warp-wide forms for the issuing warp: every lane executes them with the
// same operands and one elected lane (the same one each time: the lowest)
// acts, so no lane branches off around the tensor-core instructions.
__device__ __forceinline__ void tc_mma_elect(uint32_t d, uint64_t a, uint64_t b, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p, e;\n\tsetp.ne.u32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(kTcIdesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_commit_elect(unsigned long long *bar)
{
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(su32(bar))
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_n_elect(unsigned long long *b, uint32_t n)
{
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t@e mbarrier.arrive.shared.b64 _, [%0], %1;\n\t}" ::"r"(
            su32(b)),
        "r"(n)
        : "memory");
}

// A down tile of the tensor-memory phase: rows [pos, pos + nr) of the CTA's
// flattened (slot, row) range, within one slot and at most 128 rows. Each
// slot's part of the range starts with its remainder (length mod 128), then
// whole tiles: a short tile costs a whole tile's products, and first they run
// while the whole tiles' weights are still arriving.
__device__ __forceinline__ int tc_tile_rows(int pos, int end)
{
    const int left = min(end, (pos / kH + 1) * kH) - pos;
    const int r = left % kTcRows;
    return r ? r : kTcRows;
}

// Named barrier of the MMA warps (the producer never joins).
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory"); }

__device__ __forceinline__ float4 ldcg4(const float *p) { return __ldcg(reinterpret_cast<const float4 *>(p)); }

// 16-byte load for polling another CTA's stores: volatile asm, so every
// iteration of a polling loop issues it (a plain load may be hoisted out of
// the loop), relaxed at GPU scope (served by L2, never a stale L1 line).
__device__ __forceinline__ float4 ld_poll4(const float *p)
{
    float4 v;
    asm volatile("ld.relaxed.gpu.global.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}

__device__ __forceinline__ float ld_poll1(const float *p)
{
    float v;
    asm volatile("ld.relaxed.gpu.global.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
    return v;
}

// 4-byte asynchronous global -> shared copy and the wait for all of a thread's copies.
__device__ __forceinline__ void cp_async4(float *dst, const float *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(su32(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// all but the most recently committed group of this thread's copies have landed
__device__ __forceinline__ void cp_async_wait_group1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

__device__ __forceinline__ void mma_e4m3(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Power-of-two scale S with max|v| * S < 256 (S = 1 for an all-zero slice).
__device__ __forceinline__ float term_scale(float amax)
{
    if (!(amax > 0.0f) || !isfinite(amax))
        return 1.0f;
    int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFF) - 126;  // amax in [2^(e-1), 2^e)
    e = max(e, -118);                                                      // subnormal maxima: S <= 2^126
    return exp2f(static_cast<float>(8 - e));
}

// Writes 16 values as kTerms E4M3 terms: term t holds the E4M3 rounding of
// y_t, with y_0 = v * S and y_{t+1} = (y_t - term_t) * 16 (exact in fp32),
// so sum_t term_t / (S * 16^t) = v up to 2^-(4 kTerms) relative. b[t][j] packs
// elements 4j..4j+3 (element 4j in the low byte).
__device__ __forceinline__ void split_terms16(const float (&v)[16], float S, uint32_t (&b)[kTerms][4])
{
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float y[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            y[i] = v[4 * j + i] * S;
#pragma unroll
        for (int t = 0; t < kTerms; ++t) {
            const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(y[0], y[1]), __NV_SATFINITE, __NV_E4M3);
            const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(y[2], y[3]), __NV_SATFINITE, __NV_E4M3);
            b[t][j] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
            if (t + 1 < kTerms) {
                const float2 dl = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(lo, __NV_E4M3)));
                const float2 dh = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(hi, __NV_E4M3)));
                y[0] = (y[0] - dl.x) * 16.0f;
                y[1] = (y[1] - dl.y) * 16.0f;
                y[2] = (y[2] - dh.x) * 16.0f;
                y[3] = (y[3] - dh.y) * 16.0f;
            }
        }
    }
}

struct Terms16 {
    uint32_t w[kTerms][4];
};

// Out-of-line form of split_terms16 (one copy of the code for all callers).
__device__ __noinline__ Terms16 split16(float4 a, float4 b, float4 c, float4 d, float S)
{
    const float v[16] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w, c.x, c.y, c.z, c.w, d.x, d.y, d.z, d.w};
    Terms16 t;
    split_terms16(v, S, t.w);
    return t;
}

__device__ __forceinline__ void split16_into(const float (&v)[16], float S, uint32_t (&b)[kTerms][4])
{
    const Terms16 t = split16(make_float4(v[0], v[1], v[2], v[3]), make_float4(v[4], v[5], v[6], v[7]),
                              make_float4(v[8], v[9], v[10], v[11]), make_float4(v[12], v[13], v[14], v[15]), S);
#pragma unroll
    for (int k = 0; k < kTerms; ++k)
#pragma unroll
        for (int j = 0; j < 4; ++j)
            b[k][j] = t.w[k][j];
}

// Max over the 4 lanes that share a token (lane = 4 g + q).
__device__ __forceinline__ float quad_max(float v)
{
    v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, 1));
    return fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, 2));
}

__device__ __forceinline__ float quad_sum(float v)
{
    v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
    return v + __shfl_xor_sync(0xFFFFFFFFu, v, 2);
}


// ---------------------------------------------------------------- work plans
// Both the producer and the consumers walk the same sequence of ring stages.

struct Range {
    int begin, end;
};

__device__ __forceinline__ Range split(long long total, int part, int parts)
{
    return Range{static_cast<int>(total * part / parts), static_cast<int>(total * (part + 1) / parts)};
}

// Gate/up tiles (8 row pairs each) of the grid in one list: tiles 0..87 are
// the shared expert's, then routed slot u's tile t is 88 (u + 1) + t. CTA c
// takes tiles c, c + G, c + 2 G, ...: its tile k has list index c + k G (the
// shared tile, if any, is its tile 0). Every expert's tiles are spread over
// the whole grid, so an expert early in the list has all of its activations
// written early in the gate/up phase, and the down rows that read them need
// not wait for the slowest CTA's last tiles.
constexpr int kGuTiles = kF / 8;   // 88 tiles per expert

// S = slots of the layer: U routed experts + the always-on parts.
__device__ __forceinline__ int gu_tile_count(int S, int cta, int G)
{
    const int total = S * kGuTiles;
    return cta < total ? (total - 1 - cta) / G + 1 : 0;
}

// Gate/up tiles of the CTAs before `cta` (the first total % G CTAs take one more).
__device__ __forceinline__ unsigned gu_tiles_before(int S, int cta, int G)
{
    const unsigned total = static_cast<unsigned>(S) * kGuTiles;
    return static_cast<unsigned>(cta) * (total / G) + min(static_cast<unsigned>(cta), total % G);
}

// Down rows of one CTA, in 16-row tiles, dealt so that gate/up and down work
// together are even: a gate/up tile (8 row pairs of 2816 bytes) counts as 3
// down tiles (16 rows of 704 bytes; measured stage times are about 1 : 0.3),
// and a CTA with one more gate/up tile than another gets 3 fewer down tiles.
// Cumulative over CTAs: 16 (units(c) - 3 * gate/up tiles before c).
__device__ __forceinline__ Range down_rows(int S, int cta, int G)
{
    // 32-bit arithmetic: S * 440 * G < 2^32 for S <= 67, G <= 152 * 1000
    constexpr unsigned kW = 3;
    const unsigned units = static_cast<unsigned>(S) * (kW * kGuTiles + kH / 16);
    const unsigned c0 = cta, c1 = cta + 1;
    const int b = static_cast<int>(units * c0 / G - kW * gu_tiles_before(S, cta, G));
    const int e = static_cast<int>(units * c1 / G - kW * gu_tiles_before(S, cta + 1, G));
    return Range{16 * b, 16 * e};
}

struct DownStages {
    int begin, end;   // CTA range in the flattened (slot, row) space
    int k0, n, rot;   // first 64-row block, number of blocks, rotation
    __device__ DownStages(int S, int cta, int G)
    {
        const Range r = down_rows(S, cta, G);
        begin = r.begin;
        end = r.end;
        constexpr int kBlk = kDownTiles * 16;   // 64 rows
        constexpr int kBlocksPerSlot = kH / kBlk;
        const int first = (begin / kH) * kBlocksPerSlot + (begin % kH) / kBlk;
        const int last = end > begin ? ((end - 1) / kH) * kBlocksPerSlot + ((end - 1) % kH) / kBlk : first - 1;
        k0 = first;
        n = last - first + 1;
        rot = n > 0 ? (cta * 7) % n : 0;
    }
    // i-th stage in visiting order: absolute position and row count
    __device__ void get(int i, int &pos, int &nv) const { at(k0 + (i + rot) % n, pos, nv); }
    // stage of 64-row block k
    __device__ void at(int k, int &pos, int &nv) const
    {
        constexpr int kBlk = kDownTiles * 16;
        constexpr int kBlocksPerSlot = kH / kBlk;
        const int start = (k / kBlocksPerSlot) * kH + (k % kBlocksPerSlot) * kBlk;
        pos = max(begin, start);
        nv = min(end, start + kBlk) - pos;
    }
};

// Loads the 64 activation values (4 chunks x 16) a consumer thread owns for
// token g in K-slice `warp` of a 2816-wide row: positions 256 w + 64 c + 16 q + i.
__device__ __forceinline__ void load_slice_f32(const float *row, int warp, int q, float (&v)[4][16])
{
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const float *p = row + 256 * warp + 64 * c + 16 * q;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float4 f = ldcg4(p + 4 * k);
            v[c][4 * k + 0] = f.x;
            v[c][4 * k + 1] = f.y;
            v[c][4 * k + 2] = f.z;
            v[c][4 * k + 3] = f.w;
        }
    }
}

__device__ __forceinline__ void load_slice_bf16(const uint16_t *row, int warp, int q, float (&v)[4][16])
{
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint16_t *p = row + 256 * warp + 64 * c + 16 * q;
        const uint4 a = *reinterpret_cast<const uint4 *>(p);
        const uint4 b = *reinterpret_cast<const uint4 *>(p + 8);
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float2 f = bf16x2_to_f32(w[k]);
            v[c][2 * k] = f.x;
            v[c][2 * k + 1] = f.y;
        }
    }
}

// Gate/up ring stage: 16 smem rows (8 gate + 8 up) of 2816 bytes; warp w
// multiplies its 256-byte K-slice by the activation terms b and leaves the
// 16 x 8 partial (terms combined) in `out`.
// A-fragment words of one gate/up or lm_head stage for warp w: chunk c of
// rows g and g + 8 of the slot (bytes 256 w + 64 c + 16 q).
__device__ __forceinline__ void load_a_wide(const uint8_t *slot, int warp, int g, int q, uint4 (&ra)[4], uint4 (&rb)[4])
{
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        ra[c] = lds128(slot + g * kRowStride + 256 * warp + 64 * c + 16 * q);
        rb[c] = lds128(slot + (g + 8) * kRowStride + 256 * warp + 64 * c + 16 * q);
    }
}

// Packed activation columns. An mma B fragment (k32 x n8) carries 8 columns
// and each column is one (token, term) pair, so NB = 2 blocks hold the 15
// columns of M <= 5 tokens x 3 terms and NB = 3 blocks the 24 of M <= 8.
// Column c = 2 c' + e of block j holds
//   block 0: token c', term e
//   block 1: e = 0: token c', term 2
//            e = 1: NB = 2: token 4, term c' (c' < 3; c' = 3 is empty)
//                   NB = 3: token c' + 4, term 0
//   block 2: token c' + 4, term 1 + e (NB = 3)
// A thread's accumulator columns 2q, 2q + 1 of all blocks then cover every
// term of token q and of its second token q2 (4, split over lanes q < 3, when
// NB = 2; q + 4 when NB = 3). tok = -1 marks an empty column.
template <int NB>
__device__ __forceinline__ void column_of(int j, int c, int &tok, int &term)
{
    const int cc = c >> 1, e = c & 1;
    if (j == 0) {
        tok = cc;
        term = e;
    } else if (j == 1) {
        if (e == 0) {
            tok = cc;
            term = 2;
        } else if (NB == 2) {
            tok = cc < 3 ? 4 : -1;
            term = cc;
        } else {
            tok = cc + 4;
            term = 0;
        }
    } else {
        tok = cc + 4;
        term = 1 + e;
    }
}

// Term weights of a thread's columns: fa[t] = 16^-t / S(q), fb[t] = 16^-t / S(q2)
// (NB = 3), fb[0] = 16^-q / S(4) (NB = 2); 0 for tokens >= M.
template <int NB>
__device__ __forceinline__ void column_weights(float sa, float sb, int q, int M, float (&fa)[3], float (&fb)[3])
{
    float f = 1.0f;
#pragma unroll
    for (int t = 0; t < 3; ++t) {
        fa[t] = q < M ? f / sa : 0.0f;
        fb[t] = (NB == 3 && q + 4 < M) ? f / sb : 0.0f;
        f *= 0.0625f;
    }
    if (NB == 2)
        fb[0] = (q < 3 && 4 < M) ? (q == 0 ? 1.0f : q == 1 ? 0.0625f : 0.00390625f) / sb : 0.0f;
}

// Combines the terms of a thread's packed accumulators into
// {row r: token q, row r: token q2, row r + 8: token q, row r + 8: token q2}.
template <int NB>
__device__ __forceinline__ float4 combine_terms(const float (&acc)[NB][4], const float (&fa)[3], const float (&fb)[3])
{
    float4 r;
    r.x = acc[0][0] * fa[0] + acc[0][1] * fa[1] + acc[1][0] * fa[2];
    r.z = acc[0][2] * fa[0] + acc[0][3] * fa[1] + acc[1][2] * fa[2];
    if constexpr (NB == 2) {
        // token 4: this lane's column holds its term q; sum the quad's terms
        r.y = quad_sum(acc[1][1] * fb[0]);
        r.w = quad_sum(acc[1][3] * fb[0]);
    } else {
        r.y = acc[1][1] * fb[0] + acc[2][0] * fb[1] + acc[2][1] * fb[2];
        r.w = acc[1][3] * fb[0] + acc[2][2] * fb[1] + acc[2][3] * fb[2];
    }
    return r;
}

// Gate/up products of one 16-row tile (rows 0..7 gate, 8..15 up) over warp w's
// 256-byte K-slice with packed activation columns; returns the combined
// partial {gate q, gate q2, up q, up q2} of row g.
template <int NB>
__device__ __forceinline__ float4 gu_products_packed(const uint4 (&ra)[4], const uint4 (&rb)[4],
                                                     const uint32_t (&b)[4][NB][4], const float (&fa)[3],
                                                     const float (&fb)[3])
{
    float acc[NB][4];
#pragma unroll
    for (int j = 0; j < NB; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e)
            acc[j][e] = 0.0f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint32_t a0[4] = {ra[c].x, rb[c].x, ra[c].y, rb[c].y};
        const uint32_t a1[4] = {ra[c].z, rb[c].z, ra[c].w, rb[c].w};
#pragma unroll
        for (int j = 0; j < NB; ++j)
            mma_e4m3(acc[j], a0, b[c][j][0], b[c][j][1]);
#pragma unroll
        for (int j = 0; j < NB; ++j)
            mma_e4m3(acc[j], a1, b[c][j][2], b[c][j][3]);
    }
    return combine_terms<NB>(acc, fa, fb);
}

// E4M3 terms of 4 values (see split_terms16): w[t] packs term t of y[0..3].
__device__ __forceinline__ void split_terms4(float (&y)[4], uint32_t (&w)[kTerms])
{
#pragma unroll
    for (int t = 0; t < kTerms; ++t) {
        const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(y[0], y[1]), __NV_SATFINITE, __NV_E4M3);
        const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(y[2], y[3]), __NV_SATFINITE, __NV_E4M3);
        w[t] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
        if (t + 1 < kTerms) {
            const float2 dl = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(lo, __NV_E4M3)));
            const float2 dh = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(hi, __NV_E4M3)));
            y[0] = (y[0] - dl.x) * 16.0f;
            y[1] = (y[1] - dl.y) * 16.0f;
            y[2] = (y[2] - dh.x) * 16.0f;
            y[3] = (y[3] - dh.y) * 16.0f;
        }
    }
}

// Gate/up epilogue of one reduced tile: the lane holds gate (x, y) and up
// (z, w) of one row for its tokens a and b; writes act = comb *
// gelu_tanh(s_g g) * (s_u u) at dst_a / dst_b.
__device__ __noinline__ void gu_epilogue(float *dst_a, float *dst_b, float4 f, float sg, float su, float ca,
                                         float cb, bool ta, bool tb)
{
    if (ta)
        __stcg(dst_a, gelu_tanh(sg * f.x) * (su * f.z) * ca);
    if (tb)
        __stcg(dst_b, gelu_tanh(sg * f.y) * (su * f.w) * cb);
}

// Down epilogue of one reduced tile: adds s_d * partial into the residual
// rows h_a (token a) and h_b (token b): x, y at row r, z, w at row r + 8.
__device__ __forceinline__ void down_epilogue(float *h_a, float *h_b, float4 f, float sd0, float sd1, bool r1ok,
                                              bool ta, bool tb)
{
    if (ta) {
        atomicAdd(h_a, f.x * sd0);
        if (r1ok)
            atomicAdd(h_a + 8, f.z * sd1);
    }
    if (tb) {
        atomicAdd(h_b, f.y * sd0);
        if (r1ok)
            atomicAdd(h_b + 8, f.w * sd1);
    }
}

// Sum of the 11 K-slice partials of lane ln of tile t:
// (row ln/4, cols 2(ln%4), 2(ln%4)+1) in x, y and row ln/4 + 8 in z, w.
__device__ __forceinline__ float4 red_sum4(const Smem &s, int b, int t, int ln)
{
    float4 v = s.red[b][0][t][ln];
#pragma unroll
    for (int w = 1; w < kMW; ++w) {
        const float4 f = s.red[b][w][t][ln];
        v.x += f.x;
        v.y += f.y;
        v.z += f.z;
        v.w += f.w;
    }
    return v;
}

// Writes the pending marker into an activation buffer (tokens < M): every
// slot if n_used == 0, else the first n_used slots and the shared one. Thread
// `first` of `stride` cooperating threads; out of line (cold code).
__device__ __noinline__ void mark_act_pending(float *base, int n_used, int ns, int M, int first, int stride)
{
    const float4 pend4 = make_float4(__uint_as_float(kActPending), __uint_as_float(kActPending),
                                     __uint_as_float(kActPending), __uint_as_float(kActPending));
    const int rows = (n_used == 0 ? kMaxSlotsAll : n_used + ns) * M;
    for (int i = first; i < rows * (kF / 4); i += stride) {
        const int r = i / (kF / 4), c4 = i % (kF / 4);
        const int slot = n_used == 0 ? r / M : (r / M < n_used ? r / M : kSharedSlot + r / M - n_used);
        __stcg(reinterpret_cast<float4 *>(base + ((size_t)slot * kMaxM + r % M) * kF) + c4, pend4);
    }
}

// Packed down-phase B fragments of one expert slot for this warp's 64-wide
// K-slice, out of line (called once per slot and layer).
template <int NB>
struct DownCols {
    uint32_t b[NB][4];
    float fa[3], fb[3];
};

// act_slot: the slot's activations [token][704]. Token g's 16 values (lanes
// 4g..4g+3) are polled until no value carries the pending marker (bounded by
// the deadline; on timeout the abort flag and status are set and zeros used),
// split into terms under a power-of-two scale, and moved into the packed
// columns (column g of block j from lane 4 token + q).
template <int NB>
__device__ __noinline__ DownCols<NB> down_columns(const float *act_slot, int M, int warp, int lane, int *abort,
                                                  long long deadline, int32_t *status, int aslot)
{
    const int g = lane >> 2, q = lane & 3;
    float v[16];
    if (g < M) {
        const float *ar = act_slot + (size_t)g * kF + 64 * warp + 16 * q;
        for (int it = 0;; ++it) {
            bool ready = true;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float4 f = ld_poll4(ar + 4 * k);
                v[4 * k] = f.x;
                v[4 * k + 1] = f.y;
                v[4 * k + 2] = f.z;
                v[4 * k + 3] = f.w;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i)
                ready = ready && __float_as_uint(v[i]) != kActPending;
            if (ready)
                break;
            if ((it & 15) == 15 && (*reinterpret_cast<volatile int *>(abort) || gtime() > deadline)) {
                *reinterpret_cast<volatile int *>(abort) = 1;
                if (atomicOr(status, FGM_STATUS_WAIT_TIMEOUT) == 0) {
                    status[1] = 7;
                    status[2] = blockIdx.x;
                    status[3] = warp;
                    status[4] = aslot;
                }
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    v[i] = 0.0f;
                break;
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i)
            v[i] = 0.0f;
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i)
        amax = fmaxf(amax, fabsf(v[i]));
    const float S = term_scale(quad_max(amax));
    uint32_t T[kTerms][4];
    split16_into(v, S, T);
    DownCols<NB> r;
#pragma unroll
    for (int j = 0; j < NB; ++j) {
        int tok, term;
        column_of<NB>(j, g, tok, term);
        const bool ok = tok >= 0 && tok < M;
        const int src = 4 * (tok >= 0 ? tok : 0) + q;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t w0 = __shfl_sync(0xFFFFFFFFu, T[0][k], src);
            const uint32_t w1 = __shfl_sync(0xFFFFFFFFu, T[1][k], src);
            const uint32_t w2 = __shfl_sync(0xFFFFFFFFu, T[2][k], src);
            r.b[j][k] = ok ? (term == 0 ? w0 : term == 1 ? w1 : w2) : 0u;
        }
    }
    const int qb = NB == 2 ? 4 : q + 4;
    const float sa = __shfl_sync(0xFFFFFFFFu, S, 4 * q);
    const float sb = __shfl_sync(0xFFFFFFFFu, S, 4 * qb);
    column_weights<NB>(sa, sb, q, M, r.fa, r.fb);
    return r;
}

// Speculative sampling verify at temperature T = 1 / inv_t, run by the 352
// consumer threads of the last CTA once every CTA's logits z [M][V] and its
// per-token (max, sum of exp((z - max) / T)) over its contiguous vocabulary
// range are in memory. With p_i = softmax(z_i / T): draft d_i is kept while
// u_acc[i] < p_i(d_i); the first rejected position i emits an inverse-CDF
// sample, in vocabulary order, of p_i with d_i removed at u_next[i]; if all
// M - 1 drafts are kept, position M - 1 emits a sample of p_{M-1}.
// out = {accepted drafts, emitted token}. The CDF walk picks the CTA range
// from the per-CTA sums, then one of 11 sub-ranges from warp sums, then the
// row by a warp scan. Where rounding leaves the target past the last weight,
// the last row of positive weight is taken. A draft outside [0, V) has
// probability 0: it is rejected and removes nothing.
struct SampleShared {
    float mx[kMaxM], tot[kMaxM];
    float wsum[kMW];
    int wlast[kMW];
    float target, wx, base;
    int emit, excl, g, wsel, resort;
};

__device__ __noinline__ void sample_finish(const float *z, int64_t V, int M, int G, float inv_t,
                                           const float *part_max, const float *part_sum, const int32_t *draft,
                                           const float *u_acc, const float *u_next, const int32_t *arg,
                                           int32_t *out)
{
    __shared__ SampleShared sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const unsigned full = 0xFFFFFFFFu;
    // global max and total of every position
    if (warp < M) {
        float mx = -INFINITY;
        for (int c = lane; c < G; c += 32)
            mx = fmaxf(mx, __ldcg(part_max + c * kMaxM + warp));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            mx = fmaxf(mx, __shfl_xor_sync(full, mx, o));
        float tot = 0.0f;
        for (int c = lane; c < G; c += 32) {
            const float m = __ldcg(part_max + c * kMaxM + warp);
            if (m > -INFINITY)
                tot += __ldcg(part_sum + c * kMaxM + warp) * expf((m - mx) * inv_t);
        }
        tot = warp_sum(tot);
        if (lane == 0) {
            sh.mx[warp] = mx;
            sh.tot[warp] = tot;
        }
    }
    consumer_sync();
    // acceptance, position by position
    if (tid == 0) {
        int i = 0, excl = -1;
        for (; i < M - 1; ++i) {
            const int d = draft[i];
            if (d < 0 || d >= V)
                break;
            const float pd = expf((__ldcg(z + (size_t)i * V + d) - sh.mx[i]) * inv_t) / sh.tot[i];
            if (!(u_acc[i] < pd)) {
                excl = d;
                break;
            }
        }
        const float wx = excl >= 0 ? expf((__ldcg(z + (size_t)i * V + excl) - sh.mx[i]) * inv_t) : 0.0f;
        sh.emit = i;
        sh.excl = excl;
        sh.wx = wx;
        sh.target = u_next[i] * (sh.tot[i] - wx);
    }
    consumer_sync();
    const int i = sh.emit, excl = sh.excl;
    const float mx = sh.mx[i], target = sh.target, wx = sh.wx;
    const float *zi = z + (size_t)i * V;
    // the CTA range that holds the target: warp 0 scans the per-CTA sums in order
    if (warp == 0) {
        float base = 0.0f;
        int gsel = -1, glast = -1;
        float base_last = 0.0f;
        for (int c0 = 0; c0 < G && gsel < 0; c0 += 32) {
            const int c = c0 + lane;
            float sc = 0.0f;
            if (c < G) {
                const float m = __ldcg(part_max + c * kMaxM + i);
                if (m > -INFINITY)
                    sc = __ldcg(part_sum + c * kMaxM + i) * expf((m - mx) * inv_t);
                const Range r = split(V, c, G);
                if (excl >= r.begin && excl < r.end)
                    sc = fmaxf(sc - wx, 0.0f);
            }
            float inc = sc;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float n = __shfl_up_sync(full, inc, o);
                if (lane >= o)
                    inc += n;
            }
            const unsigned hit = __ballot_sync(full, sc > 0.0f && base + inc > target);
            const unsigned pos = __ballot_sync(full, sc > 0.0f);
            if (pos) {
                const int l = 31 - __clz(pos);
                glast = c0 + l;
                base_last = base + __shfl_sync(full, inc - sc, l);
            }
            if (hit) {
                const int l = __ffs(hit) - 1;
                gsel = c0 + l;
                base += __shfl_sync(full, inc - sc, l);
            } else {
                base += __shfl_sync(full, inc, 31);
            }
        }
        if (lane == 0) {
            sh.resort = gsel < 0;
            sh.g = gsel >= 0 ? gsel : glast;
            sh.base = gsel >= 0 ? base : base_last;
        }
    }
    consumer_sync();
    if (sh.g < 0) {   // no weight anywhere (every logit NaN, or all mass on the removed draft)
        if (tid == 0) {
            out[0] = i;
            out[1] = arg[i];
        }
        return;
    }
    const Range r = split(V, sh.g, G);
    const int per = (r.end - r.begin + kMW - 1) / kMW;
    const int w0 = r.begin + warp * per, w1 = min(r.end, w0 + per);
    auto weight = [&](int v) { return v == excl ? 0.0f : expf((__ldcg(zi + v) - mx) * inv_t); };
    // the sub-range of each warp: its sum and its last row of positive weight
    {
        float sum = 0.0f;
        int last = -1;
        for (int v = w0 + lane; v < w1; v += 32) {
            const float w = weight(v);
            sum += w;
            if (w > 0.0f)
                last = v;
        }
        sum = warp_sum(sum);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            last = max(last, __shfl_xor_sync(full, last, o));
        if (lane == 0) {
            sh.wsum[warp] = sum;
            sh.wlast[warp] = last;
        }
    }
    consumer_sync();
    if (tid == 0) {
        int wsel = -1;
        float base = sh.base;
        if (!sh.resort)
            for (int w = 0; w < kMW; ++w) {
                if (sh.wsum[w] > 0.0f && base + sh.wsum[w] > target) {
                    wsel = w;
                    break;
                }
                base += sh.wsum[w];
            }
        int last = -1;
        for (int w = 0; w < kMW; ++w)
            last = max(last, sh.wlast[w]);
        sh.wsel = wsel;
        sh.base = base;
        if (wsel < 0) {   // rounding put the target past the range's weight
            out[0] = i;
            out[1] = last >= 0 ? last : arg[i];
        }
    }
    consumer_sync();
    if (warp != sh.wsel)
        return;
    float base = sh.base;
    for (int v0 = w0; v0 < w1; v0 += 32) {
        const int v = v0 + lane;
        const float w = v < w1 ? weight(v) : 0.0f;
        float inc = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float n = __shfl_up_sync(full, inc, o);
            if (lane >= o)
                inc += n;
        }
        const unsigned hit = __ballot_sync(full, w > 0.0f && base + inc > target);
        if (hit) {
            if (lane == 0) {
                out[0] = i;
                out[1] = v0 + __ffs(hit) - 1;
            }
            return;
        }
        base += __shfl_sync(full, inc, 31);
    }
    if (lane == 0) {   // rounding between the warp's sum and its scan
        out[0] = i;
        out[1] = sh.wlast[warp];
    }
}

// Always-on part pp of a layer (its slot kSharedSlot + pp): with NS = 1 the
// layer's shared expert (expert kShared), with NS = 3 part pp of the dense
// MLP in Params::dense (gate/up rows pp * 704 .., down columns pp * 704 .. of
// its 2112-wide rows, the down rows' full-width scales).
template <int NS>
struct Parts {
    __device__ static const uint8_t *gate(const fgm_layer &L, const DenseArgs &d, int pp)
    {
        return NS > 1 ? d.gq + (size_t)pp * kF * kH : L.gate_q + (size_t)kShared * kF * kH;
    }
    __device__ static const uint8_t *up(const fgm_layer &L, const DenseArgs &d, int pp)
    {
        return NS > 1 ? d.uq + (size_t)pp * kF * kH : L.up_q + (size_t)kShared * kF * kH;
    }
    __device__ static const float *gate_s(const fgm_layer &L, const DenseArgs &d, int pp)
    {
        return NS > 1 ? d.gs + (size_t)pp * kF : L.gate_s + (size_t)kShared * kF;
    }
    __device__ static const float *up_s(const fgm_layer &L, const DenseArgs &d, int pp)
    {
        return NS > 1 ? d.us + (size_t)pp * kF : L.up_s + (size_t)kShared * kF;
    }
    // row j of the part's down matrix (kF bytes) and the row stride
    __device__ static const uint8_t *down_row(const fgm_layer &L, const DenseArgs &d, int pp, int j)
    {
        return NS > 1 ? d.dq + (size_t)j * (NS * kF) + (size_t)pp * kF : L.down_q + ((size_t)kShared * kH + j) * kF;
    }
    __device__ static const float *down_s(const fgm_layer &L, const DenseArgs &d, int pp)
    {
        return NS > 1 ? d.ds : L.down_s + (size_t)kShared * kH;
    }
};

// NB: packed column blocks (2: M <= 5, 3: M <= 8). TRACE: the phase-trace
// profiling aid is compiled in (a separate instantiation, so that the
// production kernels carry none of its code). NS: always-on parts per layer
// (1: the shared expert; 3: a 2112-wide dense MLP in every layer). TCD: the down
// phase on tcgen05 (NB = 2, NS = 1; tensor maps in Params::dmap).
template <int NB, bool TRACE, int NS = 1, bool TCD = false>
__global__ void __launch_bounds__(kThreads, 1) k_fused(const __grid_constant__ ParamsFor<NS> p)
{
    static_assert(!TCD || (NB == 2 && (NS == 1 || NS == 3)), "the tensor-memory down phase covers M <= 5");
    // the shared-memory block starts 1024-byte aligned (swizzled TMA boxes in the ring)
    extern __shared__ __align__(128) uint8_t smem_raw[];
    Smem &s = *reinterpret_cast<Smem *>(smem_raw + ((1024u - (su32(smem_raw) & 1023u)) & 1023u));
    const int G = gridDim.x, cta = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, q = lane & 3;
    const int M = p.M;
    const Ws &ws = p.ws;
    int32_t *status = ws.status;
    const long long deadline = gtime() + p.timeout_ns;
    const bool is_mma = warp < kMW;

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&s.full[i], 1);
            mbar_init(&s.empty[i], kMW);
        }
        mbar_init(&s.route, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s.tfull[i], 1);
            mbar_init(&s.tempty[i], 4);
        }
        mbar_init(&s.mdone, 1);
        mbar_init(&s.bready, 5);
        s.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    const int n_layers = p.mode == kModeLayer ? 1 : p.mode == kModeLmHead ? 0 : p.n_layers;

    // ============================================================ producer
    if (warp == kProdWarp) {
        if (lane == 0) {
            uint32_t stage = 0;
            bool ok = true;
            const uint64_t pol = l2_evict_first();
            long long *pdetail = (TRACE && p.trace && cta == G / 2)
                                     ? p.trace + (size_t)(n_layers * kTracePoints + 2) * G : nullptr;
            int p_layer = 0;
            uint32_t p_stage0 = 0;
            uint32_t p_tiles = 0;   // tensor-memory down tiles (and end markers) announced
            // Claims the next ring slot for `bytes` of copies; returns its base.
            auto claim = [&](uint32_t bytes) -> uint8_t * {
                const int slot = stage % kStages;
                if (stage >= kStages && ok)
                    ok = mbar_wait(&s.empty[slot], ((stage / kStages) - 1) & 1, s, deadline, status, 1, (int)stage);
                if (!ok)
                    return nullptr;
                mbar_expect_tx(&s.full[slot], bytes);
                if (pdetail && stage - p_stage0 < kTraceStages)
                    pdetail[((size_t)p_layer * kTraceStages + (stage - p_stage0)) * kTraceDetail] = clock64();
                return s.ring[slot];
            };
            // rows i .. i + nv - 1 of one gate/up pair of matrices ([704][2816] each)
            auto gu_rows = [&](const uint8_t *gbase, const uint8_t *ubase, int i, int nv) {
                uint8_t *dst = claim(2u * nv * kH);
                if (!dst)
                    return;
                const uint8_t *gsrc = gbase + (size_t)i * kH;
                const uint8_t *usrc = ubase + (size_t)i * kH;
                for (int rr = 0; rr < nv; ++rr) {
                    bulk_g2s_stream(dst + rr * kRowStride, gsrc + (size_t)rr * kH, kH, &s.full[stage % kStages], pol);
                    bulk_g2s_stream(dst + (8 + rr) * kRowStride, usrc + (size_t)rr * kH, kH, &s.full[stage % kStages],
                                    pol);
                }
                ++stage;
            };
            const bool lm_phase = p.mode == kModeVerify || p.mode == kModeLmHead;
            const Range rvoc = lm_phase ? split(p.V, cta, G) : Range{0, 0};
            for (int l = 0; l < n_layers && ok; ++l) {
                const fgm_layer &L = p.layers[l];
                p_layer = l;
                p_stage0 = stage;
                // router CTAs: the layer's kRouterRows router rows (and their bias
                // entries when the bias is 16-byte aligned) as the layer's first stage
                if (cta >= G - kRouterCtas) {
                    const int e0 = kRouterRows * (cta - (G - kRouterCtas));
                    const bool bias = L.router_b && (reinterpret_cast<uintptr_t>(L.router_b) & 15u) == 0;
                    constexpr uint32_t kRowsBytes = kRouterRows * kH * sizeof(uint16_t);
                    uint8_t *dst = claim(kRowsBytes + (bias ? kE * sizeof(float) : 0u));
                    if (!dst)
                        break;
                    bulk_g2s(dst, L.router_w + (size_t)e0 * kH, kRowsBytes, &s.full[stage % kStages]);
                    if (bias)
                        bulk_g2s(dst + kRowsBytes, L.router_b, kE * sizeof(float), &s.full[stage % kStages]);
                    ++stage;
                    // the next layer's rows into L2 now: their copy is issued near the
                    // end of this layer, when HBM is busiest
                    if (l + 1 < n_layers)
                        prefetch_l2(p.layers[l + 1].router_w + (size_t)e0 * kH, kRowsBytes);
                }
                // the always-on tiles (list indices below NS * kGuTiles) before the
                // routing is known, then the routed ones
                int k = 0;
                for (; cta + k * G < NS * kGuTiles && ok; ++k) {
                    const int x = cta + k * G;
                    gu_rows(Parts<NS>::gate(L, p.dense[l], x / kGuTiles), Parts<NS>::up(L, p.dense[l], x / kGuTiles),
                            8 * (x % kGuTiles), 8);
                }
                if (!ok)
                    break;
                ok = mbar_wait(&s.route, l & 1, s, deadline, status, 2, l);
                if (!ok)
                    break;
                const int pb = l & 1;
                const int U = s.n_unique[pb];
                const int n_gu = gu_tile_count(U + NS, cta, G);
                for (; k < n_gu && ok; ++k) {
                    const int x = cta + k * G - NS * kGuTiles;
                    const size_t e = s.experts[pb][x / kGuTiles];
                    gu_rows(L.gate_q + e * kF * kH, L.up_q + e * kF * kH, 8 * (x % kGuTiles), 8);
                }
                if constexpr (TCD) {
                    // Whole 128-row tiles (a slot is 22 of them), taken one at a time
                    // from a per-slot counter shared by the CTAs whose static ranges
                    // touch the slot (their home slots, whose activation terms they
                    // prepare): a CTA that runs ahead takes more of its slots' tiles.
                    // Each tile: three K-stages of two 128-byte boxes (K 640..767
                    // reads zeros past 704), its 128 row scales with the first. Then
                    // an empty stage with an end marker.
                    const DownStages dsp(U + NS, cta, G);
                    const int hs0 = dsp.begin / kH;
                    const int n_home = dsp.end > dsp.begin ? (dsp.end - 1) / kH - hs0 + 1 : 0;
                    unsigned *cnt = ws.sync + kSyncTileCount + (l & 1) * kSyncTileStride;
                    for (int h2 = 0; h2 < n_home && ok; ++h2) {
                        const int si = hs0 + h2;
                        const int e = si < U ? s.experts[pb][si] : kShared;
                        const float *dsc = si < U ? L.down_s + (size_t)e * kH : Parts<NS>::down_s(L, p.dense[l], si - U);
                        // a dense part's tile: its 704 bytes of the dense down rows
                        const CUtensorMap *dmap = &p.dmap[l];
                        int x0 = 0, y0 = e * kH;
                        if constexpr (NS > 1) {
                            if (si >= U) {
                                dmap = &p.dmap_dense[l];
                                x0 = kF * (si - U);
                                y0 = 0;
                            }
                        }
                        for (;;) {
                            const unsigned t = atomicAdd(cnt + si, 1u);
                            if (t >= static_cast<unsigned>(kH / kTcRows))
                                break;
                            const int row = static_cast<int>(t) * kTcRows;
                            s.tinfo[p_tiles % kTcInfo] = make_int2(si * kH + row, h2);
                            float *sc = &s.sc_d[(p_tiles % kTcInfo) * kTcRows];
                            ++p_tiles;
                            for (int ks = 0; ks < kTcStagesPerTile && ok; ++ks) {
                                uint8_t *dst = claim(2u * kTcBoxBytes + (ks == 0 ? kTcRows * 4u : 0u));
                                if (!dst)
                                    break;
                                const uint32_t d0 = su32(dst);
                                if (ks == 0)
                                    bulk_g2s(sc, dsc + row, kTcRows * 4u, &s.full[stage % kStages]);
                                for (int b = 0; b < 2; ++b)
                                    tma_2d(d0 + b * kTcBoxBytes, dmap, x0 + 256 * ks + 128 * b, y0 + row,
                                           &s.full[stage % kStages], pol);
                                ++stage;
                            }
                            if (!ok)
                                break;
                        }
                    }
                    if (ok) {
                        s.tinfo[p_tiles % kTcInfo] = make_int2(-1, 0);
                        ++p_tiles;
                        if (claim(0u))
                            ++stage;
                    }
                } else {
                    const DownStages dsp(U + NS, cta, G);
                    for (int di = 0; di < dsp.n && ok; ++di) {
                        int pos, nv;
                        dsp.get(di, pos, nv);
                        const int slot = pos / kH, row = pos % kH;
                        {
                            uint8_t *dst = claim(static_cast<uint32_t>(nv) * kF);
                            if (!dst)
                                break;
                            if (NS == 1 || slot < U) {
                                // 4-row (2816-byte) pieces: many mid-sized copies keep more
                                // requests in flight than one 45 KB copy
                                const uint8_t *src =
                                    slot < U ? L.down_q + ((size_t)s.experts[pb][slot] * kH + row) * kF
                                             : Parts<NS>::down_row(L, p.dense[l], 0, row);
                                for (int r4 = 0; r4 < nv; r4 += 4)
                                    bulk_g2s_stream(dst + r4 * kF, src + (size_t)r4 * kF,
                                                    static_cast<uint32_t>(min(4, nv - r4)) * kF, &s.full[stage % kStages],
                                                    pol);
                            } else {
                                // a dense part's rows are kF-byte pieces of wider rows
                                for (int rr = 0; rr < nv; ++rr)
                                    bulk_g2s_stream(dst + rr * kF, Parts<NS>::down_row(L, p.dense[l], slot - U, row + rr),
                                                    kF, &s.full[stage % kStages], pol);
                            }
                            ++stage;
                        }
                    }
                }
            }
            if (ok && lm_phase) {
                for (int v0 = rvoc.begin; v0 < rvoc.end && ok; v0 += 16) {
                    const int nv = min(16, rvoc.end - v0);
                    for (int half = 0; half < 2 && ok; ++half) {
                        uint8_t *dst = claim(static_cast<uint32_t>(nv) * kH);
                        if (!dst)
                            break;
                        const uint8_t *src = reinterpret_cast<const uint8_t *>(p.emb + (size_t)v0 * kH) + half * kH;
                        for (int rr = 0; rr < nv; ++rr)
                            bulk_g2s_stream(dst + rr * kRowStride, src + (size_t)rr * 2 * kH, kH, &s.full[stage % kStages],
                                            pol);
                        ++stage;
                    }
                }
            }
            // Every issued copy must land before the CTA may exit.
            const uint32_t first = stage > kStages ? stage - kStages : 0;
            for (uint32_t k = first; k < stage; ++k)
                for (int it = 0; it < (1 << 20); ++it)
                    if (mbar_try(&s.full[k % kStages], (k / kStages) & 1))
                        break;
        }
        return;
    }

    // ============================================================ consumers
    if constexpr (TCD) {
        // tensor memory for the down phase's two accumulators (one CTA per SM)
        if (warp == 0) {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&s.tmem_base)),
                         "r"(kTcTmemCols)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        }
    }
    uint32_t tc_tiles = 0;    // tensor-memory down tiles finished by this CTA (barrier phases)
    uint32_t tc_layers = 0;   // tensor-memory down phases run (phases of s.bready)
    uint32_t mdone_phase = 0; // phase parity of s.mdone (the issuing thread: one commit, one wait per phase)
    uint32_t stage = 0;   // ring stages consumed
    unsigned bar_target = 0;
    unsigned *bar_ctr = ws.sync;

    // Grid-wide barrier of the consumer warps (the producer never joins: it only
    // reads weights). Release-add then acquire-spin on one counter in the
    // workspace; bounded by the kernel's deadline.
    auto grid_barrier = [&]() {
        consumer_sync();
        if (tid == 0) {
            bar_target += G;
            asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(bar_ctr) : "memory");
            if (!*reinterpret_cast<volatile int *>(&s.abort)) {
                for (int it = 0;; ++it) {
                    unsigned v;
                    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(bar_ctr) : "memory");
                    if (v >= bar_target)
                        break;
                    if ((it & 63) == 63 && gtime() > deadline) {
                        s.abort = 1;
                        if (atomicOr(status, FGM_STATUS_WAIT_TIMEOUT) == 0) {
                            status[1] = 6;
                            status[2] = cta;
                            status[3] = (int)v;
                            status[4] = (int)bar_target;
                        }
                        break;
                    }
                }
            }
        }
        consumer_sync();
    };
    // Bounded exit of a warp's polling loop, the same answer in every lane: true
    // once the CTA has aborted or the kernel's deadline has passed (then the
    // abort flag, the status bit and the wait report are set).
    auto poll_give_up = [&](int site, int index) -> bool {
        int give_up = 0;
        if (lane == 0) {
            give_up = *reinterpret_cast<volatile int *>(&s.abort) != 0;
            if (!give_up && gtime() > deadline) {
                give_up = 1;
                *reinterpret_cast<volatile int *>(&s.abort) = 1;
                if (atomicOr(status, FGM_STATUS_WAIT_TIMEOUT) == 0) {
                    status[1] = site;
                    status[2] = cta;
                    status[3] = warp;
                    status[4] = index;
                }
            }
        }
        return __shfl_sync(0xFFFFFFFFu, give_up, 0) != 0;
    };

    long long *detail = (TRACE && p.trace && cta == G / 2)
                            ? p.trace + (size_t)(n_layers * kTracePoints + 2) * G : nullptr;
    int cur_layer = 0;
    uint32_t layer_stage0 = 0;
    auto dstamp = [&](uint32_t k, uint32_t k0, int which) {
        if (detail && k - k0 < kTraceStages)
            detail[((size_t)cur_layer * kTraceStages + (k - k0)) * kTraceDetail + which] = clock64();
    };
    // MMA warps: wait for the next ring stage (false after an abort) and release it
    auto stage_wait = [&]() -> bool {
        if (tid == 0)
            dstamp(stage, layer_stage0, 5);
        const bool ok = mbar_wait(&s.full[stage % kStages], (stage / kStages) & 1, s, deadline, status, 3, (int)stage);
        if (tid == 0)
            dstamp(stage, layer_stage0, 1);
        return ok;
    };
    auto stage_release = [&]() {
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&s.empty[stage % kStages]);
        if (tid == 0)
            dstamp(stage, layer_stage0, 3);
        ++stage;
    };
    uint32_t bx[4][NB][4];   // packed activation columns of this warp's K-slice (gate/up)
    float fa_x[3], fb_x[3];  // their term weights
    int cur_pb = 0;               // routing buffer of the current layer
    float *act_cur = ws.act;      // activation buffer of the current layer (alternates)
    // Activation buffers carry a pending marker until their rows are written
    // (the down rows poll for it). mark_pending(buf, n_used) marks buffer buf
    // for tokens < M: every slot if n_used == 0, else the first n_used slots and
    // the shared one. The caller guarantees that no reader of the buffer's
    // previous contents is left and that its next writers come after a grid
    // barrier.
    auto mark_pending = [&](int buf, int n_used) {
        mark_act_pending(ws.act + (size_t)buf * kMaxSlotsAll * kMaxM * kF, n_used, NS, M, cta * kConsumers + tid,
                         G * kConsumers);
    };
    // lm_head: lanes 0..3 keep the running best of tokens 2 lane, 2 lane + 1
    // over the tiles this warp reduces
    float best_v[2] = {-INFINITY, -INFINITY};
    int best_i[2] = {0x7FFFFFFF, 0x7FFFFFFF};
    float run_s[2] = {0.0f, 0.0f};   // sampling: sum of exp((z - best_v) / T) over the same tiles

    // Epilogue of one reduced tile. Expert tiles (packed columns): the lane
    // holds row r0 = lane / 4 in x, y and row r0 + 8 in z, w for its tokens
    // qa = lane % 4 and qb. lm_head tiles: token columns n0 = 2 (lane % 4), n0 + 1.
    auto finish_tile = [&](auto kind_tag, const int4 &m, int tl, const float4 &f) {
        const int r0 = lane >> 2, n0 = (lane & 3) * 2;
        constexpr int kind = decltype(kind_tag)::value;
        if constexpr (kind == kTileGateUp) {
            // m.x >> 2 = act slot, m.y = first row, m.z = row pairs | (k0 << 8), m.w = comb slot or -1;
            // x, y: gate of row r0; z, w: up of row r0 (the tile's rows 8.. are the up rows)
            // lane: row r0, tokens qa = lane % 4 and qb (packed columns)
            const int aslot = m.x >> 2, i = m.y, nv = m.z & 0xFF, k0 = m.z >> 8;
            const int qa = lane & 3, qb = NB == 2 ? 4 : qa + 4;
            if (r0 < nv) {
                const float sg = s.sc_g[k0 + r0], su = s.sc_u[k0 + r0];
                const float ca = m.w >= 0 ? s.comb[cur_pb][m.w][qa] : 1.0f;
                const float cb = m.w >= 0 ? s.comb[cur_pb][m.w][qb] : 1.0f;
                float *base = act_cur + (size_t)aslot * kMaxM * kF + i + r0;
                gu_epilogue(base + qa * kF, base + qb * kF, f, sg, su, ca, cb, qa < M,
                            qb < M && (NB == 3 || qa == 0));
            }
        } else if constexpr (kind == kTileDown) {
            // tile tl of a 64-row stage: m.y = first output row j of the stage, m.z = scale
            // index of that row, m.w = valid rows of the stage
            const int j = m.y + 16 * tl, k0 = m.z + 16 * tl, nv = m.w - 16 * tl;
            const int qa = lane & 3, qb = NB == 2 ? 4 : qa + 4;
            if (r0 < nv) {
                const float sd0 = s.sc_d[k0 + r0];
                const float sd1 = r0 + 8 < nv ? s.sc_d[k0 + r0 + 8] : 0.0f;
                down_epilogue(ws.h + (size_t)qa * kH + j + r0, ws.h + (size_t)qb * kH + j + r0, f, sd0, sd1,
                              r0 + 8 < nv, qa < M, qb < M && (NB == 3 || qa == 0));
            }
        } else {
            // m.y = first vocabulary row v0, m.z = valid rows
            const int v0 = m.y, nv = m.z;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const float za = c ? f.y : f.x, zb = c ? f.w : f.z;
                const bool ca = r0 < nv && n0 + c < M && !isnan(za);
                const bool cb = r0 + 8 < nv && n0 + c < M && !isnan(zb);
                float bz = ca ? za : -INFINITY;
                int bi = ca ? v0 + r0 : 0x7FFFFFFF;
                if (cb && better(zb, v0 + r0 + 8, bz, bi)) {
                    bz = zb;
                    bi = v0 + r0 + 8;
                }
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) {
                    const float oz = __shfl_xor_sync(0xFFFFFFFFu, bz, o);
                    const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
                    if (better(oz, oi, bz, bi)) {
                        bz = oz;
                        bi = oi;
                    }
                }
                if (p.z) {
                    // sampling: the logits go out, and the tile's sum of exp((z - bz) / T)
                    // (bz = the column's tile maximum, the same in its 8 lanes) joins the
                    // running sum kept relative to best_v
                    const int t = n0 + c;
                    if (t < M) {
                        float *zr = p.z + (size_t)t * p.V + v0;
                        if (r0 < nv)
                            zr[r0] = za;
                        if (r0 + 8 < nv)
                            zr[r0 + 8] = zb;
                    }
                    float e = (ca ? expf((za - bz) * p.inv_t) : 0.0f) + (cb ? expf((zb - bz) * p.inv_t) : 0.0f);
                    e += __shfl_xor_sync(0xFFFFFFFFu, e, 4);
                    e += __shfl_xor_sync(0xFFFFFFFFu, e, 8);
                    e += __shfl_xor_sync(0xFFFFFFFFu, e, 16);
                    if (bz > best_v[c])
                        run_s[c] = run_s[c] * expf((best_v[c] - bz) * p.inv_t) + e;
                    else if (bz > -INFINITY)
                        run_s[c] += e * expf((bz - best_v[c]) * p.inv_t);
                }
                if (better(bz, bi, best_v[c], best_i[c])) {
                    best_v[c] = bz;
                    best_i[c] = bi;
                }
            }
        }
    };

    // The partials of nt <= 2 tiles meet in shared memory buffer rbuf; after
    // one barrier, nt reducer warps (rotating over the posts) sum one tile each
    // and apply its epilogue while the other warps go on to their next
    // products. The buffers alternate: a buffer is written again only after the
    // next post's barrier, which its reducers reach after they are done. Every
    // read of an epilogue's results is preceded by a barrier (the next post's
    // or a grid barrier's).
    int rbuf = 0;
    int rot = 0;   // first reducer warp of the next post
    auto post = [&](auto kind_tag, const int4 &m0, const int4 &m1, const float (&part)[2][4], int nt, int t_off,
                    bool last_of_stage) {
#pragma unroll
        for (int t = 0; t < 2; ++t)
            if (t < nt)
                s.red[rbuf][warp][t][lane] = make_float4(part[t][0], part[t][1], part[t][2], part[t][3]);
        consumer_sync();
        int t = warp - rot;
        if (t < 0)
            t += kMW;
        if (t < nt)
            finish_tile(kind_tag, t ? m1 : m0, t_off + t, red_sum4(s, rbuf, t, lane));
        rbuf ^= 1;
        rot = rot + 1 == kMW ? 0 : rot + 1;
        if (tid == 0 && last_of_stage)
            dstamp(stage - 1, layer_stage0, 4);
    };
    auto exchange1 = [&](auto kind_tag, const int4 &m, float x, float y, float z, float w) {
        float part[2][4];
        part[0][0] = x;
        part[0][1] = y;
        part[0][2] = z;
        part[0][3] = w;
        post(kind_tag, m, m, part, 1, 0, true);
    };

    // One gate/up tile (rows i..i+nv-1 of one expert, written to act slot
    // aslot): act[aslot][n][i + ii] = comb * gelu_tanh(s_g g) * (s_u u).
    // Products of the gate/up tile at the ring head into part (the caller
    // posts tiles in pairs: one exchange barrier per two ring stages).
    auto gu_tile = [&](float (&part)[4]) {
        uint4 ra[4], rb[4];
        const bool got = stage_wait();
#pragma unroll
        for (int e = 0; e < 4; ++e)
            part[e] = 0.0f;
        if (got) {
            load_a_wide(s.ring[stage % kStages], warp, g, q, ra, rb);
            const float4 f = gu_products_packed<NB>(ra, rb, bx, fa_x, fb_x);
            part[0] = f.x;
            part[1] = f.y;
            part[2] = f.z;
            part[3] = f.w;
        }
        stage_release();
        if (tid == 0)
            dstamp(stage - 1, layer_stage0, 2);
    };

    for (int l = 0; l < n_layers; ++l) {
        const fgm_layer &L = p.layers[l];
        const int pb = l & 1;
        auto stamp = [&](int k) {
            if (TRACE && p.trace && tid == 0)
                p.trace[((size_t)l * kTracePoints + k) * G + cta] = gtime();
        };
        cur_layer = l;
        cur_pb = pb;
        act_cur = ws.act + (size_t)(l & 1) * kMaxSlotsAll * kMaxM * kF;
        layer_stage0 = stage;
        if (detail && tid == 0)
            detail[((size_t)l * kTraceStages) * kTraceDetail + 7] = clock64();
        stamp(0);
        if (p.debug_stall == l + 1 && tid == 0)
            bar_target += 1;   // the next grid barrier can never complete
        if constexpr (TCD) {
            // The down-tile counters: at layer 0 this layer's (whatever an earlier
            // launch left, even one that gave up), and at every layer the next
            // layer's (last used two layers ago, by producers that finished before
            // this layer began). The grid barrier after phase A orders these
            // stores before any tile is taken.
            if (cta == 0 && tid < kSyncTileStride) {
                ws.sync[kSyncTileCount + ((l + 1) & 1) * kSyncTileStride + tid] = 0u;
                if (l == 0)
                    ws.sync[kSyncTileCount + tid] = 0u;
            }
        }
        if (p.debug_stall == l + 1)
            grid_barrier();
        // -------------------------------------------------------- phase A
        // this CTA's always-on tiles: list indices cta, cta + G, ... below NS * kGuTiles
        const int n_sh = cta < NS * kGuTiles ? (NS * kGuTiles - 1 - cta) / G + 1 : 0;
        {
            const bool from_x = (p.mode == kModeLayer) || l == 0;
            const bool norm = p.mode != kModeLayer;
            const bool router_cta = cta >= G - kRouterCtas;
            const int e0 = kRouterRows * (cta - (G - kRouterCtas));   // first router row (router CTAs)
            // only the router CTAs and those hosting term-split units read h here;
            // token t's units sit on CTAs G - kRouterCtas - 1 - 2 t (K-slices 0..5)
            // and G - kRouterCtas - 2 - 2 t (slices 6..10), next to the router CTAs,
            // so that the two jobs run side by side and each SM converts about half
            // a row
            const int term_c = G - kRouterCtas - 1 - cta;
            const int term_t = term_c >> 1;
            const bool need_h = router_cta || (term_c >= 0 && term_t < M);
            // Lane (g, q) holds 64 values of token g in warp w's 256-wide K-slice: fp32
            // rows at positions 256 w + 64 c + 16 k + 4 q + i (v[c][4 k + i]), bf16 rows
            // at 256 w + 64 c + 32 k + 8 q + i (v[c][8 k + i]); the four lanes of a token
            // read contiguous 64 bytes at a time.
            float v[4][16];
            if (g < M && need_h) {
                if (from_x) {
                    const uint16_t *xr = p.x + (size_t)g * kH + 256 * warp + 8 * q;
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int k = 0; k < 2; ++k) {
                            const uint4 a = *reinterpret_cast<const uint4 *>(xr + 64 * c + 32 * k);
                            const uint32_t wd[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const float2 f = bf16x2_to_f32(wd[j]);
                                v[c][8 * k + 2 * j] = f.x;
                                v[c][8 * k + 2 * j + 1] = f.y;
                            }
                        }
                } else {
                    const float *hr = ws.h + (size_t)g * kH + 256 * warp + 4 * q;
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const float4 f = ldcg4(hr + 64 * c + 16 * k);
                            v[c][4 * k] = f.x;
                            v[c][4 * k + 1] = f.y;
                            v[c][4 * k + 2] = f.z;
                            v[c][4 * k + 3] = f.w;
                        }
                }
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        v[c][i] = 0.0f;
            }
            // scales of this CTA's shared-expert gate/up rows, copied asynchronously;
            // each thread waits for its copies before the first gate/up tile, and
            // the exchange barrier that follows makes them visible to the reducers
            for (int i = tid; i < 8 * n_sh; i += kConsumers) {
                const int x = cta + (i >> 3) * G, pp = x / kGuTiles, row = 8 * (x % kGuTiles) + (i & 7);
                cp_async4(&s.sc_g[kMaxGuRows + i], Parts<NS>::gate_s(L, p.dense[l], pp) + row);
                cp_async4(&s.sc_u[kMaxGuRows + i], Parts<NS>::up_s(L, p.dense[l], pp) + row);
            }
            cp_async_commit();
            if (l == 0) {
                // residual (stack) or accumulator (layer) initialisation, split over CTAs
                for (int i = cta * kConsumers + tid; i < kMaxM * kH; i += G * kConsumers) {
                    const int n = i / kH;
                    float init = 0.0f;
                    if (p.mode != kModeLayer && n < M)
                        init = bf16_to_f32(p.x[i]);
                    ws.h[i] = init;
                }
            }
            // router bias of a CTA whose bias entries were not copied with its rows
            const bool bias_copied = L.router_b && (reinterpret_cast<uintptr_t>(L.router_b) & 15u) == 0;
            float rbias = 0.0f;
            if (router_cta && tid < kRouterRows * M && L.router_b && !bias_copied)
                rbias = __ldg(L.router_b + e0 + tid / M);
            {
                // sum of squares and the router dot products on the un-normalised
                // row; RMSNorm is a per-token scale, applied to the dots afterwards
                float ss = 0.0f, dot[kRouterRows];
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        ss += v[c][i] * v[c][i];
#pragma unroll
                for (int j = 0; j < kRouterRows; ++j)
                    dot[j] = 0.0f;
                if (router_cta) {
                    // the layer's router rows arrive as this CTA's first ring stage
                    const bool got = stage_wait();
                    const uint8_t *slot = s.ring[stage % kStages];
                    if (got) {
#pragma unroll
                        for (int j = 0; j < kRouterRows; ++j) {
                            const uint16_t *wr = reinterpret_cast<const uint16_t *>(slot) + j * kH + 256 * warp;
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                if (from_x) {
#pragma unroll
                                    for (int k = 0; k < 2; ++k) {
                                        const uint4 w4 = *reinterpret_cast<const uint4 *>(wr + 64 * c + 32 * k + 8 * q);
                                        const uint32_t w8[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                                        for (int m = 0; m < 4; ++m) {
                                            const float2 f = bf16x2_to_f32(w8[m]);
                                            dot[j] += f.x * v[c][8 * k + 2 * m] + f.y * v[c][8 * k + 2 * m + 1];
                                        }
                                    }
                                } else {
#pragma unroll
                                    for (int k = 0; k < 4; ++k) {
                                        const uint2 w2 = *reinterpret_cast<const uint2 *>(wr + 64 * c + 16 * k + 4 * q);
                                        const float2 f0 = bf16x2_to_f32(w2.x), f1 = bf16x2_to_f32(w2.y);
                                        dot[j] += f0.x * v[c][4 * k] + f0.y * v[c][4 * k + 1] + f1.x * v[c][4 * k + 2] +
                                                  f1.y * v[c][4 * k + 3];
                                    }
                                }
                            }
                        }
                        if (bias_copied && tid < kRouterRows * M)
                            rbias = reinterpret_cast<const float *>(slot + kRouterRows * kH * sizeof(uint16_t))[e0 + tid / M];
                    }
                    stage_release();
                }
                ss = quad_sum(ss);
#pragma unroll
                for (int j = 0; j < kRouterRows; ++j)
                    dot[j] = quad_sum(dot[j]);
                if (q == 0) {
                    s.part[warp][g] = ss;
#pragma unroll
                    for (int j = 0; j < kRouterRows; ++j)
                        s.part2[j][warp][g] = dot[j];
                }
                stamp(1);
            }
            consumer_sync();
            stamp(2);
            {
                if (router_cta && tid < kRouterRows * M) {
                    const int j = tid / M, t = tid % M;
                    float z = 0.0f, tot = 0.0f;
#pragma unroll
                    for (int w = 0; w < kMW; ++w) {
                        z += s.part2[j][w][t];
                        tot += s.part[w][t];
                    }
                    const float rt = norm ? 1.0f / sqrtf(tot / static_cast<float>(kH) + kEps) : 1.0f;
                    __stcg(ws.logits + t * kE + e0 + j, z * rt + rbias);
                }
                // Activation terms of the gate/up products, computed once per grid:
                // unit (token t, 256-wide K-slice w) is split by warp w of one of
                // token t's two term CTAs (it holds the slice in lanes 4 t .. 4 t + 3),
                // 8 values a lane after a pass through shared memory (the exchange
                // buffer is idle in phase A), into kTerms E4M3 terms under a
                // power-of-two scale per unit.
                const int t = term_t;
                if (term_c >= 0 && t < M && (warp < 6) == ((term_c & 1) == 0)) {
                    const int w = warp;
                    const int k0 = 256 * w + 8 * lane;
                    float *sx = reinterpret_cast<float *>(&s.red[0][0][0][0]) + 256 * warp;
                    if (g == t) {
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            if (from_x) {
#pragma unroll
                                for (int k = 0; k < 2; ++k) {
                                    float4 *d = reinterpret_cast<float4 *>(sx + 64 * c + 32 * k + 8 * q);
                                    d[0] = make_float4(v[c][8 * k], v[c][8 * k + 1], v[c][8 * k + 2], v[c][8 * k + 3]);
                                    d[1] = make_float4(v[c][8 * k + 4], v[c][8 * k + 5], v[c][8 * k + 6], v[c][8 * k + 7]);
                                }
                            } else {
#pragma unroll
                                for (int k = 0; k < 4; ++k)
                                    *reinterpret_cast<float4 *>(sx + 64 * c + 16 * k + 4 * q) =
                                        make_float4(v[c][4 * k], v[c][4 * k + 1], v[c][4 * k + 2], v[c][4 * k + 3]);
                            }
                        }
                    }
                    __syncwarp();
                    float xv[8];
                    {
                        const float4 a = *reinterpret_cast<const float4 *>(sx + 8 * lane);
                        const float4 b = *reinterpret_cast<const float4 *>(sx + 8 * lane + 4);
                        xv[0] = a.x; xv[1] = a.y; xv[2] = a.z; xv[3] = a.w;
                        xv[4] = b.x; xv[5] = b.y; xv[6] = b.z; xv[7] = b.w;
                    }
                    float r = 1.0f;
                    if (norm) {
                        float tot = 0.0f;
#pragma unroll
                        for (int w2 = 0; w2 < kMW; ++w2)
                            tot += s.part[w2][t];
                        r = 1.0f / sqrtf(tot / static_cast<float>(kH) + kEps);
                    }
                    float amax = 0.0f;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        xv[i] *= r;
                        amax = fmaxf(amax, fabsf(xv[i]));
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1)
                        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
                    const float S = term_scale(amax);
                    uint32_t w0[kTerms], w1[kTerms];
                    float y0[4] = {xv[0] * S, xv[1] * S, xv[2] * S, xv[3] * S};
                    float y1[4] = {xv[4] * S, xv[5] * S, xv[6] * S, xv[7] * S};
                    split_terms4(y0, w0);
                    split_terms4(y1, w1);
#pragma unroll
                    for (int tt = 0; tt < kTerms; ++tt)
                        __stcg(reinterpret_cast<uint2 *>(ws.xterms + ((size_t)t * kTerms + tt) * kH + k0),
                               make_uint2(w0[tt], w1[tt]));
                    if (lane == 0)
                        __stcg(ws.xscale + t * kMW + w, S);
                }
            }
        }
        if (l == 0)
            mark_pending(0, 0);   // this layer's buffer (the next one is marked after its down rows)
        stamp(3);
        stamp(4);
        grid_barrier();
        stamp(5);
        // -------------------------------------------------------- phase B
        {
            float lv[4];
            if (warp < M) {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    lv[k] = __ldcg(ws.logits + warp * kE + lane + 32 * k);
            }
            if (warp < M) {
                // top-8 by repeated warp argmax (ties to the lower index)
                bool bad = false;
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    if (isnan(lv[k])) {
                        lv[k] = -INFINITY;
                        bad = true;
                    }
                if (__any_sync(0xFFFFFFFFu, bad) && lane == 0)
                    atomicOr(status, FGM_STATUS_NONFINITE_LOGITS);
                // top-8 (larger logit first, ties to the lower index): each round
                // takes the largest remaining key with one redux.sync max, then the
                // lowest index holding it. Keys order floats as unsigned integers;
                // 0 marks a taken logit (-inf maps to 0x007FFFFF, still above it).
                uint32_t key[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t b = __float_as_uint(lv[k]);
                    key[k] = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
                }
                uint32_t top_key = 0, my_key = 0;
                int my_i = 0;
#pragma unroll 1
                for (int rr = 0; rr < kK; ++rr) {
                    const uint32_t lk = max(max(key[0], key[1]), max(key[2], key[3]));
                    const uint32_t gk = __reduce_max_sync(0xFFFFFFFFu, lk);
                    unsigned bal[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        bal[k] = __ballot_sync(0xFFFFFFFFu, key[k] == gk);
                    const int kw = bal[0] ? 0 : bal[1] ? 1 : bal[2] ? 2 : 3;
                    const unsigned bw = kw == 0 ? bal[0] : kw == 1 ? bal[1] : kw == 2 ? bal[2] : bal[3];
                    const int lw = __ffs(bw) - 1;
                    if (lane == lw) {
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            if (k == kw)
                                key[k] = 0u;
                    }
                    if (rr == 0)
                        top_key = gk;
                    if (rr == lane) {
                        my_key = gk;
                        my_i = lw + 32 * kw;
                    }
                }
                const auto key_value = [](uint32_t kk) {
                    return __uint_as_float((kk & 0x80000000u) ? (kk & 0x7FFFFFFFu) : ~kk);
                };
                const float top0 = key_value(top_key), my_v = key_value(my_key);
                // lanes 0..7 hold the 8 picks; weights = exp(l - l_max) / sum
                const float ex = lane < kK ? (top0 == -INFINITY ? 1.0f : expf(my_v - top0)) : 0.0f;
                float z = ex;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    z += __shfl_xor_sync(0xFFFFFFFFu, z, o);
                if (lane < kK) {
                    s.tk_ids[warp][lane] = my_i;
                    s.tk_w[warp][lane] = ex / z;
                }
            }
            // gate/up B fragments of this warp's K-slice: column g of each block
            // (packed (token, term) columns), loaded once the top-k is done: their
            // L2 traffic would slow the top-k down
            {
#pragma unroll
                for (int j = 0; j < NB; ++j) {
                    int tok, term;
                    column_of<NB>(j, g, tok, term);
                    const bool ok = tok >= 0 && tok < M;
                    const uint8_t *src = ws.xterms + ((size_t)(ok ? tok : 0) * kTerms + term) * kH + 256 * warp + 16 * q;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint4 w4 = make_uint4(0u, 0u, 0u, 0u);
                        if (ok)
                            w4 = __ldcg(reinterpret_cast<const uint4 *>(src + 64 * c));
                        bx[c][j][0] = w4.x;
                        bx[c][j][1] = w4.y;
                        bx[c][j][2] = w4.z;
                        bx[c][j][3] = w4.w;
                    }
                }
                // the scales of this lane's tokens; the weights are formed after the
                // top-k, so that nothing waits for these loads before then
                const int qb = NB == 2 ? 4 : q + 4;
                fa_x[0] = q < M ? __ldcg(ws.xscale + q * kMW + warp) : 1.0f;
                fb_x[0] = qb < M ? __ldcg(ws.xscale + qb * kMW + warp) : 1.0f;
            }
            stamp(10);
            for (int i = tid; i < kE; i += kConsumers)
                s.mark[i] = 0;
            consumer_sync();
            if (tid < M * kK)
                s.mark[s.tk_ids[tid >> 3][tid & 7]] = 1;
            consumer_sync();
            if (warp == 0) {
                int base = 0;
#pragma unroll
                for (int k = 0; k < kE / 32; ++k) {
                    const int e = 32 * k + lane;
                    const bool m = s.mark[e] != 0;
                    const unsigned bal = __ballot_sync(0xFFFFFFFFu, m);
                    const int pos = base + __popc(bal & ((1u << lane) - 1u));
                    if (m) {
                        s.experts[pb][pos] = e;
                        s.slot_of[e] = pos;
                    }
                    base += __popc(bal);
                }
                if (lane == 0)
                    s.n_unique[pb] = base;
            }
            for (int i = tid; i < kMaxSlotsAll * 8; i += kConsumers)
                s.comb[pb][i >> 3][i & 7] = 0.0f;
            consumer_sync();
            stamp(11);
            if (tid < M * kK) {
                const int t = tid >> 3, rr = tid & 7;
                s.comb[pb][s.slot_of[s.tk_ids[t][rr]]][t] = s.tk_w[t][rr];
                if (cta == 0 && p.ids) {
                    const size_t base = p.mode == kModeLayer ? 0 : (size_t)l * M * kK;
                    p.ids[base + tid] = s.tk_ids[t][rr];
                    if (p.mode == kModeLayer && p.wts)
                        p.wts[tid] = s.tk_w[t][rr];
                }
            }
            consumer_sync();
            if (tid == 0)
                mbar_arrive(&s.route);
            stamp(6);
            const int U = s.n_unique[pb];
            const int n_gu = gu_tile_count(U + NS, cta, G);
            // row scales of this CTA's routed gate/up rows and of its down rows,
            // copied asynchronously (cp.async); each thread waits for its copies
            // before the first routed tile, and the next exchange barrier makes
            // them visible to the reducers
            for (int k = tid; k < 8 * (n_gu - n_sh); k += kConsumers) {
                const int x = cta + (n_sh + k / 8) * G - NS * kGuTiles;
                const size_t row = (size_t)s.experts[pb][x / kGuTiles] * kF + 8 * (x % kGuTiles) + k % 8;
                cp_async4(&s.sc_g[k], L.gate_s + row);
                cp_async4(&s.sc_u[k], L.up_s + row);
            }
            if constexpr (!TCD) {
                // (the tensor-memory phase's producer copies each tile's scales)
                const Range rd = down_rows(U + NS, cta, G);
                for (int k = tid; k < rd.end - rd.begin; k += kConsumers) {
                    const int pos = rd.begin + k;
                    const int si = pos / kH;
                    const float *ds = si < U ? L.down_s + (size_t)s.experts[pb][si] * kH
                                             : Parts<NS>::down_s(L, p.dense[l], si - U);
                    cp_async4(&s.sc_d[k], ds + pos % kH);
                }
            }
            cp_async_commit();
            bool scales_ready = false;
            {
                const float sa = fa_x[0], sb = fb_x[0];
                column_weights<NB>(sa, sb, q, M, fa_x, fb_x);
            }
            // the shared expert's rows of this CTA first (their copies were issued
            // before the routing was known), then its routed rows
            float pend[2][4];
            int4 pend_m = make_int4(0, 0, 0, 0);
            bool have_pend = false;
            for (int it = 0;; ++it) {
                int aslot, i, nv, k0, cslot = -1;
                if (it == 0)
                    cp_async_wait_group1();   // the shared-expert scales (phase A's copies)
                if (!scales_ready && it >= n_sh) {
                    cp_async_wait_all();
                    scales_ready = true;
                }
                if (it >= n_gu)
                    break;
                if (it < n_sh) {
                    const int x = cta + it * G;
                    i = 8 * (x % kGuTiles);
                    nv = 8;
                    aslot = kSharedSlot + x / kGuTiles;
                    k0 = kMaxGuRows + 8 * it;
                } else {
                    const int x = cta + it * G - NS * kGuTiles;
                    const int u = x / kGuTiles;
                    i = 8 * (x % kGuTiles);
                    nv = 8;
                    aslot = u;
                    cslot = u;
                    k0 = 8 * (it - n_sh);
                }
                const int4 m = make_int4(kTileGateUp | (aslot << 2), i, nv | (k0 << 8), cslot);
                const bool last = it + 1 >= n_gu;
                if (!have_pend) {
                    gu_tile(pend[0]);
                    pend_m = m;
                    have_pend = true;
                    if (last) {
                        post(KindTag<kTileGateUp>{}, m, m, pend, 1, 0, true);
                        have_pend = false;
                    }
                } else {
                    gu_tile(pend[1]);
                    post(KindTag<kTileGateUp>{}, pend_m, m, pend, 2, 0, true);
                    have_pend = false;
                }
            }
        }
        cp_async_wait_all();   // (CTAs without routed gate/up rows: the down scales)
        stamp(7);
        // Phase C polls the activation rows it reads until the pending marker
        // is gone (no fence or counter between the phases).
        consumer_sync();
        stamp(8);
        // -------------------------------------------------------- phase C
        if constexpr (TCD) {
            const int U = s.n_unique[pb];
            const DownStages ds(U + NS, cta, G);
            const int si0 = ds.begin / kH;
            uint8_t *bop = reinterpret_cast<uint8_t *>(&s.red[0][0][0][0]);   // [2][kTcBBytes]: idle exchange buffer
            // 1. B operands of the (at most two) home slots this CTA's static range
            //    touches: token t's 704 activations of a slot are polled (16-byte
            //    loads) until none is pending, scaled by a power of two per (slot,
            //    token) and written as kTerms E4M3 terms in columns 3 t + e (the
            //    other columns stay zero). The first slot's, on which the first
            //    tile waits, by warps 2 t and 2 t + 1 (half a row each, the scale
            //    from both halves through shared memory); the second's by warp
            //    4 + t after all consumers meet, announced on s.bready, which the
            //    issuing thread waits for before that slot's first tile.
            for (int i = tid; i < 2 * kTcBBytes / 16; i += kConsumers)
                reinterpret_cast<uint4 *>(bop)[i] = make_uint4(0u, 0u, 0u, 0u);
            consumer_sync();
            constexpr int kQ = kF / 4;   // 176 float4 of a row
            // polls float4 m0 + lane + 32 jj (jj < NJ, below m1) of token t's row of home
            // slot h2, then builds those terms under the slot-token scale S
            auto tc_operand = [&](int h2, int t, int m0, int m1, auto nj, float *half_amax, int pair_bar) {
                constexpr int NJ = decltype(nj)::value;
                const int si = si0 + h2;
                const int aslot = si < U ? si : kSharedSlot + si - U;
                const float *a = act_cur + ((size_t)aslot * kMaxM + t) * kF;
                float4 v[NJ];
                for (int it = 0;; ++it) {
                    bool pending = false;
#pragma unroll
                    for (int jj = 0; jj < NJ; ++jj) {
                        const int m = m0 + lane + 32 * jj;
                        v[jj] = m < m1 ? ld_poll4(a + 4 * m) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                        pending |= __float_as_uint(v[jj].x) == kActPending || __float_as_uint(v[jj].y) == kActPending ||
                                   __float_as_uint(v[jj].z) == kActPending || __float_as_uint(v[jj].w) == kActPending;
                    }
                    if (!__any_sync(0xFFFFFFFFu, pending))
                        break;
                    if ((it & 15) == 15 && poll_give_up(11, aslot)) {
#pragma unroll
                        for (int jj = 0; jj < NJ; ++jj)
                            v[jj] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                        break;
                    }
                }
                float amax = 0.0f;
#pragma unroll
                for (int jj = 0; jj < NJ; ++jj)
                    amax = fmaxf(fmaxf(amax, fmaxf(fabsf(v[jj].x), fabsf(v[jj].y))), fmaxf(fabsf(v[jj].z), fabsf(v[jj].w)));
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
                if (half_amax) {
                    // the other half's maximum: both warps of the pair meet on their barrier
                    if (lane == 0)
                        half_amax[m0 == 0 ? 0 : 1] = amax;
                    asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory");
                    amax = fmaxf(half_amax[0], half_amax[1]);
                }
                const float S = term_scale(amax);
                if (lane == 0 && m0 == 0)
                    s.dscale[h2][t] = S;
                uint8_t *b = bop + h2 * kTcBBytes;
#pragma unroll
                for (int jj = 0; jj < NJ; ++jj) {
                    const int m = m0 + lane + 32 * jj;
                    if (m < m1) {
                        // four consecutive k: four consecutive bytes of each term column
                        float y[4] = {v[jj].x * S, v[jj].y * S, v[jj].z * S, v[jj].w * S};
                        uint32_t w[kTerms];
                        split_terms4(y, w);
#pragma unroll
                        for (int e = 0; e < kTerms; ++e)
                            *reinterpret_cast<uint32_t *>(b + tc_b_offset(3 * t + e, 4 * m)) = w[e];
                    }
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            };
            const bool has0 = ds.end > ds.begin;
            const bool has1 = has0 && ds.end > (si0 + 1) * kH;
            if (warp < 10 && has0 && (warp >> 1) < M) {
                const int t = warp >> 1, hf = warp & 1;
                tc_operand(0, t, hf * (kQ / 2), (hf + 1) * (kQ / 2), std::integral_constant<int, (kQ / 2 + 31) / 32>{},
                           s.tc_amax[t], 3 + t);
            }
            consumer_sync();
            if (warp >= 4 && warp < 9) {
                const int t = warp - 4;
                if (has1 && t < M)
                    tc_operand(1, t, 0, kQ, std::integral_constant<int, (kQ + 31) / 32>{}, nullptr, 0);
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&s.bready);
            }
            // 2. the tiles, in the order the producer took them (its tile records,
            //    then an end marker): warp kMW - 1 issues the products (one
            //    elected lane), warps 0..3 (tensor-memory lanes 32 w .. 32 w + 31)
            //    read the accumulators, combine the terms, apply the row scales and
            //    add into the residual stream. The issuing warp publishes the stage
            //    and tile counts after the phase (the tile count is known only to it).
            if (warp == kMW - 1) {
                // the whole warp runs the issuing loop and one elected lane issues
                // (measured a little faster than one lane's loop, 0.3 % per step);
                // waits agree across lanes through lane 0
                auto wait_all = [&](unsigned long long *b, uint32_t parity, int site, int index) -> bool {
                    const bool r = mbar_wait(b, parity, s, deadline, status, site, index);
                    return __shfl_sync(0xFFFFFFFFu, r ? 1 : 0, 0) != 0;
                };
                bool ok = __shfl_sync(0xFFFFFFFFu, *reinterpret_cast<volatile int *>(&s.abort) == 0 ? 1 : 0, 0) != 0;
                bool issued = false;      // products issued in this phase
                bool b1_ready = false;    // the second home slot's operand seen built
                uint32_t gt = tc_tiles;
                if (lane == 0)
                    s.tc_next = gt;   // (after an abort: where it stopped)
                __syncwarp();
                for (; ok; ++gt) {
                    const int buf = gt & 1;
                    // the epilogue has read this accumulator two tiles ago
                    if (gt >= 2 && !(ok = wait_all(&s.tempty[buf], ((gt >> 1) - 1) & 1, 8, (int)gt)))
                        break;
                    tc_fence_after();
                    const uint32_t d = s.tmem_base + static_cast<uint32_t>(buf * kTcN);
                    bool end_marker = false;
                    for (int ks = 0; ks < kTcStagesPerTile && ok; ++ks) {
                        const int slot = stage % kStages;
                        if (lane == 0)
                            dstamp(stage, layer_stage0, 5);
                        if (!(ok = wait_all(&s.full[slot], (stage / kStages) & 1, 3, (int)stage)))
                            break;
                        if (lane == 0)
                            dstamp(stage, layer_stage0, 1);
                        const int2 inf = s.tinfo[gt % kTcInfo];
                        if (inf.y == 1 && !b1_ready) {
                            if (!(ok = wait_all(&s.bready, tc_layers & 1, 12, (int)gt)))
                                break;
                            b1_ready = true;
                        }
                        if (inf.x < 0) {
                            // the end marker's empty stage: its slot back, then the
                            // epilogue told through this accumulator's barrier
                            mbar_arrive_n_elect(&s.empty[slot], kMW);
                            ++stage;
                            mbar_arrive_n_elect(&s.tfull[buf], 1);
                            end_marker = true;
                            break;
                        }
                        tc_fence_after();
                        // descriptors of the stage's first A and B blocks; the others
                        // differ in the start address field only (shared-memory
                        // addresses stay below 2^18 bytes, so the field never carries)
                        const uint64_t bdesc = __shfl_sync(0xFFFFFFFFu, tc_desc_nosw(su32(bop + inf.y * kTcBBytes)), 0);
                        const uint64_t adesc = __shfl_sync(0xFFFFFFFFu, tc_desc_sw128(su32(s.ring[slot])), 0);
                        const uint32_t du = __shfl_sync(0xFFFFFFFFu, d, 0);
#pragma unroll
                        for (int b = 0; b < 2; ++b)
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {
                                const int kg = 256 * ks + 128 * b + 32 * kk;
                                if (kg < kF)
                                    tc_mma_elect(du, adesc + static_cast<uint64_t>((b * kTcBoxBytes + kk * 32) >> 4),
                                                 bdesc + static_cast<uint64_t>((kg * 16) >> 4), kg > 0);
                            }
                        // the slot goes back to the producer when its products are
                        // done: kMW - 1 of its arrivals now, the last one the commit's
                        // (the issuing warp does not wait)
                        tc_commit_elect(&s.empty[slot]);
                        mbar_arrive_n_elect(&s.empty[slot], kMW - 1);
                        issued = true;
                        if (lane == 0) {
                            dstamp(stage, layer_stage0, 2);
                            dstamp(stage, layer_stage0, 3);
                        }
                        ++stage;
                    }
                    if (end_marker) {
                        if (lane == 0)
                            s.tc_next = gt + 1;
                        break;
                    }
                    if (ok)
                        tc_commit_elect(&s.tfull[buf]);
                }
                // every product issued is done before the phase ends (also after
                // an abort: nothing may be in flight when tensor memory is
                // released); products always finish, so the wait only counts tries
                if (issued) {
                    tc_commit_elect(&s.mdone);
                    for (int it = 0; it < (1 << 22); ++it)
                        if (__shfl_sync(0xFFFFFFFFu, mbar_try(&s.mdone, mdone_phase) ? 1 : 0, 0))
                            break;
                    mdone_phase ^= 1u;
                }
                if (lane == 0)
                    s.tc_stage = stage;
                __syncwarp();
            } else if (warp < 4) {
                for (uint32_t gt = tc_tiles;; ++gt) {
                    const int buf = gt & 1;
                    if (!mbar_wait(&s.tfull[buf], (gt >> 1) & 1, s, deadline, status, 10, (int)gt))
                        break;
                    const int2 inf = s.tinfo[gt % kTcInfo];
                    if (inf.x < 0) {
                        // the end marker: nothing to read; its phase of the
                        // accumulator's barrier is answered like a tile's
                        __syncwarp();
                        if (lane == 0)
                            mbar_arrive(&s.tempty[buf]);
                        break;
                    }
                    tc_fence_after();
                    float v[16];
                    tc_ld16(s.tmem_base + (static_cast<uint32_t>(32 * warp) << 16) + static_cast<uint32_t>(buf * kTcN), v);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&s.tempty[buf]);
                    const int r = 32 * warp + lane;
                    const int j = inf.x % kH + r;
                    const float sd = s.sc_d[(gt % kTcInfo) * kTcRows + r];
#pragma unroll
                    for (int t = 0; t < 5; ++t)
                        if (t < M)
                            atomicAdd(ws.h + (size_t)t * kH + j,
                                      (v[3 * t] + v[3 * t + 1] * 0.0625f + v[3 * t + 2] * 0.00390625f) /
                                          s.dscale[inf.y][t] * sd);
                }
            }
            consumer_sync();
            stage = s.tc_stage;
            tc_tiles = s.tc_next;
            ++tc_layers;
        } else
        {
            const int U = s.n_unique[pb];
            const DownStages ds(U + NS, cta, G);
            // A CTA's rows span at most two slots (it owns fewer than 2816 rows):
            // their activation terms (this warp's 64-wide K-slice, token g) are
            // prepared once, up front.
            const int si0 = ds.begin / kH;
            DownCols<NB> dc[2];   // packed activation columns of the (at most two) slots
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int si = si0 + h2;
                const bool slot_ok = si < U + NS && (h2 == 0 || ds.end > (si0 + 1) * kH);   // same for the whole CTA
                if (slot_ok) {
                    const int aslot = si < U ? si : kSharedSlot + si - U;
                    dc[h2] = down_columns<NB>(act_cur + (size_t)aslot * kMaxM * kF, M, warp, lane, &s.abort, deadline,
                                              status, aslot);
                } else {
#pragma unroll
                    for (int j = 0; j < NB; ++j)
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            dc[h2].b[j][k] = 0u;
#pragma unroll
                    for (int t = 0; t < 3; ++t) {
                        dc[h2].fa[t] = 0.0f;
                        dc[h2].fb[t] = 0.0f;
                    }
                }
            }
            int kk = ds.rot;   // visiting order without a division per stage
            for (int di = 0; di < ds.n; ++di) {
                int pos, nv;
                ds.at(ds.k0 + kk, pos, nv);
                kk = kk + 1 == ds.n ? 0 : kk + 1;
                const int si = pos / kH, j = pos % kH;
                const int hs = si == si0 ? 0 : 1;
                uint32_t bt[NB][4];
                float fa[3], fb[3];
#pragma unroll
                for (int jj = 0; jj < NB; ++jj)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        bt[jj][k] = hs ? dc[1].b[jj][k] : dc[0].b[jj][k];
#pragma unroll
                for (int t = 0; t < 3; ++t) {
                    fa[t] = hs ? dc[1].fa[t] : dc[0].fa[t];
                    fb[t] = hs ? dc[1].fb[t] : dc[0].fb[t];
                }
                const bool got = stage_wait();
                const uint8_t *slot = s.ring[stage % kStages];
#pragma unroll
                for (int t0 = 0; t0 < kDownTiles; t0 += 2) {
                    // a stage's rows beyond nv are skipped half by half (same for the
                    // whole CTA): a partial stage costs about its rows
                    const bool half_used = 16 * t0 < nv;
                    float po[2][4];
                    // two tiles x NB packed blocks: 2 NB independent accumulator chains
                    float acc[2][NB][4];
#pragma unroll
                    for (int t = 0; t < 2; ++t)
#pragma unroll
                        for (int jj = 0; jj < NB; ++jj)
#pragma unroll
                            for (int e2 = 0; e2 < 4; ++e2)
                                acc[t][jj][e2] = 0.0f;
                    if (got && half_used) {
                        uint4 ra[2], rb[2];
#pragma unroll
                        for (int t = 0; t < 2; ++t) {
                            ra[t] = lds128(slot + (16 * (t0 + t) + g) * kF + 64 * warp + 16 * q);
                            rb[t] = lds128(slot + (16 * (t0 + t) + g + 8) * kF + 64 * warp + 16 * q);
                        }
#pragma unroll
                        for (int step = 0; step < 2; ++step)
#pragma unroll
                            for (int t = 0; t < 2; ++t) {
                                const uint32_t a[4] = {step ? ra[t].z : ra[t].x, step ? rb[t].z : rb[t].x,
                                                       step ? ra[t].w : ra[t].y, step ? rb[t].w : rb[t].y};
#pragma unroll
                                for (int jj = 0; jj < NB; ++jj)
                                    mma_e4m3(acc[t][jj], a, bt[jj][2 * step], bt[jj][2 * step + 1]);
                            }
                    }
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        const float4 f = combine_terms<NB>(acc[t], fa, fb);
                        po[t][0] = f.x;
                        po[t][1] = f.y;
                        po[t][2] = f.z;
                        po[t][3] = f.w;
                    }
                    if (t0 + 2 == kDownTiles) {
                        if (tid == 0)
                            dstamp(stage, layer_stage0, 2);
                        stage_release();
                    }
                    // tiles t0, t0 + 1 (rows beyond the stage's nv rows are skipped)
                    if (half_used) {
                        const int4 md = make_int4(kTileDown, j, pos - ds.begin, nv);
                        post(KindTag<kTileDown>{}, md, md, po, 16 * (t0 + 1) < nv ? 2 : 1, t0, t0 + 2 == kDownTiles);
                    }
                }
            }
        }
        // The next layer writes the other buffer: mark the slots it held two
        // layers ago (all of them after layer 0). Its last readers were the down
        // rows of layer l - 1, all done before this layer began.
        if (l + 1 < n_layers)
            mark_pending((l + 1) & 1, l == 0 ? 0 : s.n_unique[(l - 1) & 1]);
        stamp(9);
        grid_barrier();
    }
    if constexpr (TCD) {
        // every product has completed (the issuing thread waited for a commit
        // after its last products of each phase)
        consumer_sync();
        if (warp == 0) {
            tc_fence_after();
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(s.tmem_base), "r"(kTcTmemCols)
                         : "memory");
        }
    }
    if (TRACE && p.trace && tid == 0)
        p.trace[((size_t)n_layers * kTracePoints) * G + cta] = gtime();

    // ------------------------------------------------------------ outputs
    if (p.mode == kModeLayer || p.mode == kModeStack) {
        for (int i = cta * kConsumers + tid; i < M * kH; i += G * kConsumers)
            p.y[i] = f32_to_bf16(__ldcg(ws.h + i));
    } else {
        // lm_head input: bf16(RMSNorm(h)) after the stack, or the given bf16 rows.
        // warp w's K-slice in each half (1408 elements) of a row: 128 w + 32 c + 8 q + [0, 8)
        uint32_t bh[2][4][4];
        if (p.mode == kModeVerify) {
            float ss = 0.0f;
            if (is_mma && g < M) {
                float v[4][16];
                load_slice_f32(ws.h + (size_t)g * kH, warp, q, v);
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        ss += v[c][i] * v[c][i];
            }
            ss = quad_sum(ss);
            if (is_mma && q == 0)
                s.part[warp][g] = ss;
            consumer_sync();
            if (is_mma) {
                float tot = 0.0f;
#pragma unroll
                for (int w = 0; w < kMW; ++w)
                    tot += s.part[w][g];
                const float r = g < M ? 1.0f / sqrtf(tot / static_cast<float>(kH) + kEps) : 0.0f;
#pragma unroll
                for (int half = 0; half < 2; ++half)
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        float hv[8];
                        if (g < M) {
                            const float *hp = ws.h + (size_t)g * kH + 1408 * half + 128 * warp + 32 * c + 8 * q;
                            const float4 f0 = ldcg4(hp), f1 = ldcg4(hp + 4);
                            hv[0] = f0.x; hv[1] = f0.y; hv[2] = f0.z; hv[3] = f0.w;
                            hv[4] = f1.x; hv[5] = f1.y; hv[6] = f1.z; hv[7] = f1.w;
                        } else {
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                hv[i] = 0.0f;
                        }
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            bh[half][c][k] = static_cast<uint32_t>(f32_to_bf16(hv[2 * k] * r)) |
                                             (static_cast<uint32_t>(f32_to_bf16(hv[2 * k + 1] * r)) << 16);
                    }
            }
        } else if (is_mma) {
#pragma unroll
            for (int half = 0; half < 2; ++half)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint4 w4 = make_uint4(0u, 0u, 0u, 0u);
                    if (g < M)
                        w4 = *reinterpret_cast<const uint4 *>(p.x + (size_t)g * kH + 1408 * half + 128 * warp + 32 * c + 8 * q);
                    bh[half][c][0] = w4.x;
                    bh[half][c][1] = w4.y;
                    bh[half][c][2] = w4.z;
                    bh[half][c][3] = w4.w;
                }
        }
        const Range rv = split(p.V, cta, G);
        for (int v0 = rv.begin; v0 < rv.end; v0 += 16) {
            const int nv = min(16, rv.end - v0);
            float acc[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint4 ra[4], rb[4];
                const bool got = stage_wait();
                if (got) {
                    load_a_wide(s.ring[stage % kStages], warp, g, q, ra, rb);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint32_t a0[4] = {ra[c].x, rb[c].x, ra[c].y, rb[c].y};
                        const uint32_t a1[4] = {ra[c].z, rb[c].z, ra[c].w, rb[c].w};
                        mma_bf16(acc[c & 1], a0, bh[half][c][0], bh[half][c][1]);
                        mma_bf16(acc[c & 1], a1, bh[half][c][2], bh[half][c][3]);
                    }
                }
                stage_release();
            }
            exchange1(KindTag<kTileLmHead>{}, make_int4(kTileLmHead, v0, nv, 0), acc[0][0] + acc[1][0], acc[0][1] + acc[1][1],
                      acc[0][2] + acc[1][2], acc[0][3] + acc[1][3]);
        }
        if (lane < 4) {
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                s.best_v[warp][2 * lane + c] = best_v[c];
                s.best_i[warp][2 * lane + c] = best_i[c];
                s.samp_s[warp][2 * lane + c] = run_s[c];
            }
        }
        consumer_sync();
        if (tid < kMaxM) {
            float bv = s.best_v[0][tid];
            int bi = s.best_i[0][tid];
#pragma unroll
            for (int w = 1; w < kMW; ++w)
                if (better(s.best_v[w][tid], s.best_i[w][tid], bv, bi)) {
                    bv = s.best_v[w][tid];
                    bi = s.best_i[w][tid];
                }
            __stcg(ws.part_val + cta * kMaxM + tid, bv);
            __stcg(ws.part_idx + cta * kMaxM + tid, bi);
            if (p.z) {
                float sum = 0.0f;
                for (int w = 0; w < kMW; ++w)
                    if (s.best_v[w][tid] > -INFINITY)
                        sum += s.samp_s[w][tid] * expf((s.best_v[w][tid] - bv) * p.inv_t);
                __stcg(ws.part_sum + cta * kMaxM + tid, sum);
            }
        }
    }
    if (TRACE && p.trace && tid == 0)
        p.trace[((size_t)n_layers * kTracePoints + 1) * G + cta] = gtime();

    // ------------------------------------------------------------ exit
    // The last CTA to get here reduces the lm_head winners (lm_head modes)
    // and returns the barrier counters to zero for the next launch: every
    // CTA has passed its last grid barrier by then.
    consumer_sync();
    if (tid == 0) {
        __threadfence();
        const unsigned done = atomicAdd(bar_ctr + 1, 1u);
        s.last = done == static_cast<unsigned>(G - 1);
    }
    consumer_sync();
    if (!s.last)
        return;
    __threadfence();
    if (p.mode == kModeVerify || p.mode == kModeLmHead) {
        __shared__ int32_t arg[kMaxM];
        if (warp < M) {
            float bv = -INFINITY;
            int bi = 0x7FFFFFFF;
            for (int c = lane; c < G; c += 32) {
                const float vv = __ldcg(ws.part_val + c * kMaxM + warp);
                const int ii = __ldcg(ws.part_idx + c * kMaxM + warp);
                if (better(vv, ii, bv, bi)) {
                    bv = vv;
                    bi = ii;
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
            if (lane == 0) {
                if (bi == 0x7FFFFFFF) {
                    bi = 0;
                    atomicOr(status, FGM_STATUS_NONFINITE_LOGITS);
                }
                arg[warp] = bi;
                if (p.argmax)
                    p.argmax[warp] = bi;
                if (p.maxlogit)
                    p.maxlogit[warp] = bv;
            }
        }
        consumer_sync();
        if (p.z) {
            if (is_mma)
                sample_finish(p.z, p.V, M, G, p.inv_t, ws.part_val, ws.part_sum, p.draft, p.u_acc, p.u_next, arg,
                              p.out);
        } else if (tid == 0 && p.mode == kModeVerify) {
            int a = 0;
            while (a < M - 1 && p.draft[a] == arg[a])
                ++a;
            p.out[0] = a;
            p.out[1] = arg[a];
        }
    }
    if (tid == 0) {
        bar_ctr[1] = 0;
        atomicExch(bar_ctr, 0u);
    }
}

}  // namespace fused
}  // namespace fgm
