// C ABI of the library (declared in include/fgm.h): argument validation,
// workspace carving and launch sequencing. Every stage of the step runs in
// the CUDA kernels of basic_kernels.cuh / fused_step.cuh / lm_head_fp8.cuh.
#include <cmath>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "basic_kernels.cuh"
#include "fused_step.cuh"
#include "lm_head_fp8.cuh"
#include "lm_head_fp8_tc.cuh"

namespace fgm {
namespace {

thread_local char g_err[512] = "";

int fail(int code, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

#define FGM_CUDA(call)                                                                         \
    do {                                                                                       \
        cudaError_t e_ = (call);                                                               \
        if (e_ != cudaSuccess)                                                                 \
            return fail(FGM_ERR_CUDA, "%s failed: %s", #call, cudaGetErrorString(e_));         \
    } while (0)

#define FGM_CHECK_LAUNCH()                                                                     \
    do {                                                                                       \
        cudaError_t e_ = cudaGetLastError();                                                   \
        if (e_ != cudaSuccess)                                                                 \
            return fail(FGM_ERR_CUDA, "kernel launch failed: %s (%s:%d)", cudaGetErrorString(e_), \
                        __FILE__, __LINE__);                                                   \
    } while (0)

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool ready = false;
    bool ok = false;
    int sms = 0;
    int fused_grid = 0;   // CTAs of the persistent kernel (one per SM), 0 if it cannot be co-resident
};

int g_path = FGM_PATH_FUSED;
long long g_timeout_ns = 2000000000LL;
// the persistent kernel's shared memory: its block plus slack to align it to 1024 bytes
constexpr size_t kFusedSmemBytes = sizeof(fused::Smem) + 1024;
long long *g_trace = nullptr;
int g_debug_stall = 0;
size_t g_trace_n = 0;
DeviceInfo g_dev[kMaxDevices];

// Checks (once per device) that the current device is an sm_103 GPU and
// raises the dynamic shared-memory limit of the kernels that need it.
int device_ready(int *sms)
{
    int dev = 0;
    FGM_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices)
        return fail(FGM_ERR_DEVICE, "device index %d out of range", dev);
    DeviceInfo &d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0;
        FGM_CUDA(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev));
        FGM_CUDA(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev));
        FGM_CUDA(cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev));
        d.ok = (major == 10 && minor == 3);
        if (d.ok) {
#define FGM_SMEM(k, bytes) FGM_CUDA(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes))
            FGM_SMEM(k_gateup_basic<1>, 1 * kH * 4);
            FGM_SMEM(k_gateup_basic<2>, 2 * kH * 4);
            FGM_SMEM(k_gateup_basic<3>, 3 * kH * 4);
            FGM_SMEM(k_gateup_basic<4>, 4 * kH * 4);
            FGM_SMEM(k_gateup_basic<5>, 5 * kH * 4);
            FGM_SMEM(k_gateup_basic<6>, 6 * kH * 4);
            FGM_SMEM(k_gateup_basic<7>, 7 * kH * 4);
            FGM_SMEM(k_gateup_basic<8>, 8 * kH * 4);
            FGM_SMEM(k_lmhead_basic<1>, 1 * kH * 4);
            FGM_SMEM(k_lmhead_basic<2>, 2 * kH * 4);
            FGM_SMEM(k_lmhead_basic<3>, 3 * kH * 4);
            FGM_SMEM(k_lmhead_basic<4>, 4 * kH * 4);
            FGM_SMEM(k_lmhead_basic<5>, 5 * kH * 4);
            FGM_SMEM(k_lmhead_basic<6>, 6 * kH * 4);
            FGM_SMEM(k_lmhead_basic<7>, 7 * kH * 4);
            FGM_SMEM(k_lmhead_basic<8>, 8 * kH * 4);
            FGM_SMEM(fp8head::k_lmhead_fp8<false>, fp8head::kSmemBytes);
            FGM_SMEM(fp8head::k_lmhead_fp8<true>, fp8head::kSmemBytes);
            FGM_SMEM(fp8tc::k_lmhead_fp8_tc<false>, fp8tc::kSmemBytes);
            FGM_SMEM(fp8tc::k_lmhead_fp8_tc<true>, fp8tc::kSmemBytes);
#undef FGM_SMEM
            const void *kerns[9] = {reinterpret_cast<const void *>(fused::k_fused<2, false>),
                                    reinterpret_cast<const void *>(fused::k_fused<3, false>),
                                    reinterpret_cast<const void *>(fused::k_fused<2, true>),
                                    reinterpret_cast<const void *>(fused::k_fused<3, true>),
                                    reinterpret_cast<const void *>(fused::k_fused<2, false, 3>),
                                    reinterpret_cast<const void *>(fused::k_fused<3, false, 3>),
                                    reinterpret_cast<const void *>(fused::k_fused<2, false, 1, true>),
                                    reinterpret_cast<const void *>(fused::k_fused<2, true, 1, true>),
                                    reinterpret_cast<const void *>(fused::k_fused<2, false, 3, true>)};
            int per_sm = 1 << 30;
            for (const void *k : kerns) {
                FGM_CUDA(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFusedSmemBytes));
                int n = 0;
                FGM_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, fused::kThreads, kFusedSmemBytes));
                per_sm = n < per_sm ? n : per_sm;
            }
            d.fused_grid = (per_sm >= 1 && d.sms >= fused::kMinCtas) ? d.sms : 0;
        }
        d.ready = true;
    }
    if (!d.ok)
        return fail(FGM_ERR_DEVICE, "device %d is not an sm_103 GPU; this library is built for sm_103a", dev);
    if (sms)
        *sms = d.sms;
    return FGM_OK;
}

int fused_grid()
{
    int dev = 0;
    FGM_CUDA(cudaGetDevice(&dev));
    const int G = g_dev[dev].fused_grid;
    if (G <= 0)
        return fail(FGM_ERR_DEVICE, "the persistent kernel cannot be resident on this device");
    return G;
}

// Launches the persistent kernel (cooperative: all CTAs co-resident).
int tc_down_map(const uint8_t *down_q, CUtensorMap *map, bool dense);

int launch_fused(fused::Params &prm, cudaStream_t st)
{
    const int G = fused_grid();
    if (G < 0)
        return G;
    // the tensor-memory path runs the down phase on tcgen05 (M <= 5, one shared expert)
    // (its bulk copies of row scales want 16-byte aligned scale arrays; else the
    // mma.sync down phase runs)
    bool tcd = (g_path == FGM_PATH_FUSED || g_path == FGM_PATH_FUSED_TC) && prm.M <= 5 &&
               (prm.dense_parts == 0 || prm.dense_parts == 3) && prm.mode != fused::kModeLmHead;
    const int n_tc = prm.mode == fused::kModeLayer ? 1 : prm.n_layers;
    for (int l = 0; tcd && l < n_tc; ++l)
        if ((reinterpret_cast<uintptr_t>(prm.layers[l].down_s) & 15u) ||
            (prm.dense_parts && ((reinterpret_cast<uintptr_t>(prm.dense[l].ds) & 15u) ||
                                 (reinterpret_cast<uintptr_t>(prm.dense[l].dq) & 15u))))
            tcd = false;
    fused::ParamsDense pd;   // the dense variant's parameter block (NS = 3)
    if (prm.dense_parts == 3)
        memset(&pd, 0, sizeof pd);
    if (tcd) {
        const int n_l = n_tc;
        for (int l = 0; l < n_l; ++l) {
            int rc = tc_down_map(prm.layers[l].down_q, &prm.dmap[l], false);
            if (rc == FGM_OK && prm.dense_parts)
                rc = tc_down_map(prm.dense[l].dq, &pd.dmap_dense[l], true);
            if (rc != FGM_OK)
                return rc;
        }
    }
    prm.timeout_ns = g_timeout_ns;
    const int n_l = prm.mode == fused::kModeLayer ? 1 : prm.mode == fused::kModeLmHead ? 0 : prm.n_layers;
    const size_t need = (size_t)(n_l * fused::kTracePoints + 2) * G + (size_t)n_l * fused::kTraceStages * fused::kTraceDetail;
    prm.trace = (g_trace && g_trace_n >= need) ? g_trace : nullptr;
    prm.debug_stall = g_debug_stall;
    g_debug_stall = 0;
    void *args[] = {&prm};
    // packed activation columns: 2 blocks of 8 hold M <= 5 tokens x 3 terms, 3 blocks M <= 8
    const bool traced = prm.trace != nullptr && prm.dense_parts == 0;
    const void *kern = prm.dense_parts == 3
                           ? (tcd ? reinterpret_cast<const void *>(fused::k_fused<2, false, 3, true>)
                              : prm.M <= 5 ? reinterpret_cast<const void *>(fused::k_fused<2, false, 3>)
                                           : reinterpret_cast<const void *>(fused::k_fused<3, false, 3>))
                       : tcd ? (traced ? reinterpret_cast<const void *>(fused::k_fused<2, true, 1, true>)
                                       : reinterpret_cast<const void *>(fused::k_fused<2, false, 1, true>))
                       : prm.M <= 5 ? (traced ? reinterpret_cast<const void *>(fused::k_fused<2, true>)
                                              : reinterpret_cast<const void *>(fused::k_fused<2, false>))
                                    : (traced ? reinterpret_cast<const void *>(fused::k_fused<3, true>)
                                              : reinterpret_cast<const void *>(fused::k_fused<3, false>));
    if (!traced)
        prm.trace = nullptr;
    if (prm.dense_parts == 3) {
        static_cast<fused::Params &>(pd) = prm;
        args[0] = &pd;
    }
    FGM_CUDA(cudaLaunchCooperativeKernel(kern, dim3(G),
                                         dim3(fused::kThreads), args, kFusedSmemBytes, st));
    return FGM_OK;
}

fused::Params fused_params(int mode, int M, const Ws &w)
{
    fused::Params prm;
    memset(&prm, 0, sizeof prm);
    prm.mode = mode;
    prm.M = M;
    prm.ws = w;
    return prm;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A dense MLP's pointers and width (index: its layer, for the message).
int check_mlp(const fgm_mlp *m, int index, DenseArgs *out)
{
    if (!m)
        return fail(FGM_ERR_INVALID_ARG, "dense MLP %d is NULL", index);
    if (m->width < kF || m->width > kMaxDense * kF || m->width % kF)
        return fail(FGM_ERR_INVALID_ARG, "dense MLP %d width %d: a multiple of %d up to %d", index, m->width, kF,
                    kMaxDense * kF);
    const void *q[] = {m->gate_q, m->up_q, m->down_q};
    const void *sc[] = {m->gate_s, m->up_s, m->down_s};
    for (int i = 0; i < 3; ++i) {
        if (!q[i] || !aligned16(q[i]))
            return fail(FGM_ERR_INVALID_ARG, "dense MLP %d: weight %d NULL or not 16-byte aligned", index, i);
        if (!sc[i] || (reinterpret_cast<uintptr_t>(sc[i]) & 3u))
            return fail(FGM_ERR_INVALID_ARG, "dense MLP %d: scale %d NULL or not 4-byte aligned", index, i);
    }
    *out = DenseArgs{m->gate_q, m->gate_s, m->up_q, m->up_s, m->down_q, m->down_s, m->width / kF};
    return FGM_OK;
}

int check_layer(const fgm_layer *L, int index)
{
    if (!L)
        return fail(FGM_ERR_INVALID_ARG, "layer %d: null layer struct", index);
    const void *ptrs[] = {L->router_w, L->gate_q, L->gate_s, L->up_q, L->up_s, L->down_q, L->down_s};
    const char *names[] = {"router_w", "gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s"};
    for (int i = 0; i < 7; ++i) {
        if (!ptrs[i])
            return fail(FGM_ERR_INVALID_ARG, "layer %d: %s is NULL", index, names[i]);
        if (!aligned16(ptrs[i]))
            return fail(FGM_ERR_INVALID_ARG, "layer %d: %s is not 16-byte aligned", index, names[i]);
    }
    if (L->router_b && (reinterpret_cast<uintptr_t>(L->router_b) & 3u))
        return fail(FGM_ERR_INVALID_ARG, "layer %d: router_b is not 4-byte aligned", index);
    return FGM_OK;
}

int check_ws(void *ws, size_t ws_bytes, int M, int64_t V)
{
    if (!ws)
        return fail(FGM_ERR_WORKSPACE, "workspace is NULL");
    if (reinterpret_cast<uintptr_t>(ws) & 255u)
        return fail(FGM_ERR_WORKSPACE, "workspace is not 256-byte aligned");
    const size_t need = fgm_workspace_bytes(M, V);
    if (ws_bytes < need)
        return fail(FGM_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", ws_bytes, need);
    return FGM_OK;
}

int check_m(int M)
{
    if (M < 1 || M > kMaxM)
        return fail(FGM_ERR_INVALID_ARG, "M = %d outside [1, %d]", M, kMaxM);
    return FGM_OK;
}

#define FGM_TRY(expr)              \
    do {                           \
        int rc_ = (expr);          \
        if (rc_ != FGM_OK)         \
            return rc_;            \
    } while (0)

template <int M>
int launch_layer_experts(const fgm_layer *L, const Ws &w, float *out, const DenseArgs &dn, cudaStream_t st)
{
    k_gateup_basic<M><<<dim3(kF / 32, kMaxSlotsAll), 256, M * kH * 4, st>>>(
        L->gate_q, L->gate_s, L->up_q, L->up_s, w.xn, w.meta, w.comb, w.act, dn);
    FGM_CHECK_LAUNCH();
    k_down_basic<M><<<dim3(kH / 32, kMaxSlotsAll), 256, 0, st>>>(L->down_q, L->down_s, w.act, w.meta, out, dn);
    FGM_CHECK_LAUNCH();
    return FGM_OK;
}

int launch_experts(int M, const fgm_layer *L, const Ws &w, float *out, const DenseArgs &dn, cudaStream_t st)
{
    switch (M) {
    case 1: return launch_layer_experts<1>(L, w, out, dn, st);
    case 2: return launch_layer_experts<2>(L, w, out, dn, st);
    case 3: return launch_layer_experts<3>(L, w, out, dn, st);
    case 4: return launch_layer_experts<4>(L, w, out, dn, st);
    case 5: return launch_layer_experts<5>(L, w, out, dn, st);
    case 6: return launch_layer_experts<6>(L, w, out, dn, st);
    case 7: return launch_layer_experts<7>(L, w, out, dn, st);
    default: return launch_layer_experts<8>(L, w, out, dn, st);
    }
}

// Router + dedup + experts of one layer reading w.xn, adding into `out`; with
// dn.parts > 0 the dense shared MLP takes the place of the shared expert.
int run_layer(int M, const fgm_layer *L, const Ws &w, float *out, int32_t *ids_out, float *w_out,
              cudaStream_t st, const DenseArgs &dn = DenseArgs{})
{
    k_router_logits<<<kE, 256, 0, st>>>(w.xn, M, L->router_w, L->router_b, w.logits);
    FGM_CHECK_LAUNCH();
    k_topk_dedup<<<1, 256, 0, st>>>(w.logits, M, dn.parts ? dn.parts : 1, w.meta, w.comb, ids_out, w_out,
                                     w.status);
    FGM_CHECK_LAUNCH();
    return launch_experts(M, L, w, out, dn, st);
}

int lmhead_grid(int sms) { return sms * 4 < kMaxParts ? sms * 4 : kMaxParts; }

template <int M>
int launch_lmhead_t(const uint16_t *emb, int64_t V, const uint16_t *hb, const Ws &w, int G, cudaStream_t st)
{
    k_lmhead_basic<M><<<G, 256, M * kH * 4, st>>>(emb, V, hb, w.part_val, w.part_idx);
    FGM_CHECK_LAUNCH();
    return FGM_OK;
}

int launch_lmhead(int M, const uint16_t *emb, int64_t V, const uint16_t *hb, const Ws &w, int G,
                  cudaStream_t st)
{
    switch (M) {
    case 1: return launch_lmhead_t<1>(emb, V, hb, w, G, st);
    case 2: return launch_lmhead_t<2>(emb, V, hb, w, G, st);
    case 3: return launch_lmhead_t<3>(emb, V, hb, w, G, st);
    case 4: return launch_lmhead_t<4>(emb, V, hb, w, G, st);
    case 5: return launch_lmhead_t<5>(emb, V, hb, w, G, st);
    case 6: return launch_lmhead_t<6>(emb, V, hb, w, G, st);
    case 7: return launch_lmhead_t<7>(emb, V, hb, w, G, st);
    default: return launch_lmhead_t<8>(emb, V, hb, w, G, st);
    }
}

int check_layers(const fgm_layer *layers, int n_layers)
{
    if (!layers)
        return fail(FGM_ERR_INVALID_ARG, "layers is NULL");
    if (n_layers < 1 || n_layers > FGM_MAX_LAYERS)
        return fail(FGM_ERR_INVALID_ARG, "n_layers = %d outside [1, %d]", n_layers, FGM_MAX_LAYERS);
    for (int l = 0; l < n_layers; ++l)
        FGM_TRY(check_layer(&layers[l], l));
    return FGM_OK;
}

int check_vocab(const uint16_t *emb, int64_t V)
{
    if (!emb || !aligned16(emb))
        return fail(FGM_ERR_INVALID_ARG, "emb is NULL or not 16-byte aligned");
    if (V < 1 || V > 0x7FFFFFFFLL)
        return fail(FGM_ERR_INVALID_ARG, "V = %lld outside [1, 2^31)", (long long)V);
    return FGM_OK;
}

int check_vocab_fp8(const uint8_t *emb_q, const float *emb_s, int64_t V)
{
    if (!emb_q || !aligned16(emb_q))
        return fail(FGM_ERR_INVALID_ARG, "emb_q is NULL or not 16-byte aligned");
    if (!emb_s || (reinterpret_cast<uintptr_t>(emb_s) & 3u))
        return fail(FGM_ERR_INVALID_ARG, "emb_s is NULL or not 4-byte aligned");
    if (V < 1 || V > 0x7FFFFFFFLL)
        return fail(FGM_ERR_INVALID_ARG, "V = %lld outside [1, 2^31)", (long long)V);
    return FGM_OK;
}

// FP8 lm_head argmax in one launch (and, with draft/out, greedy acceptance).
// h: bf16 rows, or with `norm` the fp32 residual stream to normalise first.
// cuTensorMapEncodeTiled from the driver, looked up once through the runtime.
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

int encode_tiled_fn(EncodeTiledFn *fn)
{
    static EncodeTiledFn cached = nullptr;
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    if (!cached) {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !f)
            return fail(FGM_ERR_CUDA, "cuTensorMapEncodeTiled not available from the driver");
        cached = reinterpret_cast<EncodeTiledFn>(f);
    }
    *fn = cached;
    return FGM_OK;
}

// FP8 lm_head on the tensor-memory path (fp8tc): a 2-D tensor map over the
// E4M3 rows, 128 x 128-byte boxes in the 128-byte swizzle.
int run_lmhead_fp8_tc(const uint8_t *emb_q, const float *emb_s, int64_t V, const void *h, bool norm, int M,
                      int32_t *argmax, float *maxlogit, const int32_t *draft, int32_t *out, const Ws &w, int sms,
                      cudaStream_t st)
{
    EncodeTiledFn encode = nullptr;
    FGM_TRY(encode_tiled_fn(&encode));
    CUtensorMap tmap;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kH), static_cast<cuuint64_t>(V)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kH)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(fp8tc::kChunk), static_cast<cuuint32_t>(fp8tc::kRows)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(emb_q), dims, strides,
                              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(FGM_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    fp8tc::Args a;
    a.scale = emb_s;
    a.V = static_cast<int>(V);
    a.h = h;
    a.M = M;
    a.part_val = w.part_val;
    a.part_idx = w.part_idx;
    a.done = w.sync + kSyncLmHeadDone;
    a.argmax = argmax;
    a.maxlogit = maxlogit;
    a.draft = draft;
    a.out = out;
    a.status = w.status;
    a.timeout_ns = g_timeout_ns;
    const int G = fp8tc::grid_for(V, sms);
    if (norm)
        fp8tc::k_lmhead_fp8_tc<true><<<G, fp8tc::kThreads, fp8tc::kSmemBytes, st>>>(tmap, a);
    else
        fp8tc::k_lmhead_fp8_tc<false><<<G, fp8tc::kThreads, fp8tc::kSmemBytes, st>>>(tmap, a);
    FGM_CHECK_LAUNCH();
    return FGM_OK;
}

// Tensor maps of one layer's down matrices ([129 * 2816 rows][704 bytes]), or
// with `dense` of a dense MLP's down matrix ([2816 rows][3 * 704 bytes]):
// 128 x 128-byte boxes in the 128-byte swizzle, zeros past the row's end.
// Encoded once per weight address and kept.
int tc_down_map(const uint8_t *down_q, CUtensorMap *map, bool dense)
{
    struct Entry {
        const void *ptr;
        bool dense;
        CUtensorMap map;
    };
    static Entry cache[2 * FGM_MAX_LAYERS];
    static int n = 0, next = 0;
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n; ++i)
        if (cache[i].ptr == down_q && cache[i].dense == dense) {
            *map = cache[i].map;
            return FGM_OK;
        }
    EncodeTiledFn encode = nullptr;
    FGM_TRY(encode_tiled_fn(&encode));
    Entry e;
    e.ptr = down_q;
    e.dense = dense;
    const cuuint64_t width = dense ? 3u * kF : kF;
    const cuuint64_t dims[2] = {width, dense ? static_cast<cuuint64_t>(kH) : static_cast<cuuint64_t>(kNE) * kH};
    const cuuint64_t strides[1] = {width};
    const cuuint32_t estr[2] = {1, 1};
    const cuuint32_t box[2] = {128, 128};
    const CUresult r = encode(&e.map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(down_q), dims, strides,
                              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(FGM_ERR_CUDA, "cuTensorMapEncodeTiled (down matrix) failed (%d)", static_cast<int>(r));
    const int slot = n < 2 * FGM_MAX_LAYERS ? n++ : (next++ % (2 * FGM_MAX_LAYERS));
    cache[slot] = e;
    *map = e.map;
    return FGM_OK;
}

// FP8 lm_head: the tensor-memory kernel on FGM_PATH_FUSED_TC, the mma.sync
// kernel otherwise (1.2 % faster on a GB300).
int run_lmhead_fp8(const uint8_t *emb_q, const float *emb_s, int64_t V, const void *h, bool norm, int M,
                   int32_t *argmax, float *maxlogit, const int32_t *draft, int32_t *out, const Ws &w,
                   int sms, cudaStream_t st)
{
    if (g_path == FGM_PATH_FUSED_TC)
        return run_lmhead_fp8_tc(emb_q, emb_s, V, h, norm, M, argmax, maxlogit, draft, out, w, sms, st);
    fp8head::Args a;
    a.q = emb_q;
    a.scale = emb_s;
    a.V = static_cast<int>(V);
    a.h = h;
    a.M = M;
    a.part_val = w.part_val;
    a.part_idx = w.part_idx;
    a.done = w.sync + kSyncLmHeadDone;
    a.argmax = argmax;
    a.maxlogit = maxlogit;
    a.draft = draft;
    a.out = out;
    a.status = w.status;
    const int G = fp8head::grid_for(V, sms);
    if (norm)
        fp8head::k_lmhead_fp8<true><<<G, fp8head::kThreads, fp8head::kSmemBytes, st>>>(a);
    else
        fp8head::k_lmhead_fp8<false><<<G, fp8head::kThreads, fp8head::kSmemBytes, st>>>(a);
    FGM_CHECK_LAUNCH();
    return FGM_OK;
}

// The stack on w.h (already holding the input), layer by layer.
int run_stack(const fgm_layer *layers, int n_layers, int M, const Ws &w, int32_t *ids_trace,
              cudaStream_t st, const DenseArgs *dns = nullptr)
{
    for (int l = 0; l < n_layers; ++l) {
        k_rmsnorm<<<M, 256, 0, st>>>(w.h, w.xn, nullptr);
        FGM_CHECK_LAUNCH();
        FGM_TRY(run_layer(M, &layers[l], w, w.h, ids_trace ? ids_trace + (size_t)l * M * kK : nullptr,
                          nullptr, st, dns ? dns[l] : DenseArgs{}));
    }
    return FGM_OK;
}

// The persistent kernel takes per-layer dense MLPs when all are 2112 wide.
bool dense_fused(const DenseArgs *dns, int n_layers)
{
    if (!dns)
        return true;
    for (int l = 0; l < n_layers; ++l)
        if (dns[l].parts != kMaxDense)
            return false;
    return true;
}

void set_dense(fused::Params &prm, const DenseArgs *dns, int n_layers)
{
    if (!dns)
        return;
    for (int l = 0; l < n_layers; ++l)
        prm.dense[l] = dns[l];
    prm.dense_parts = kMaxDense;
}

int verify_step_impl(const fgm_layer *layers, int n_layers, const uint16_t *emb, int64_t V,
                     const uint16_t *x, const int32_t *draft, int M, int32_t *argmax, int32_t *out,
                     void *ws, cudaStream_t st, int sms, const DenseArgs *dns = nullptr)
{
    Ws w = ws_carve(ws);
    if (g_path != FGM_PATH_STAGED && dense_fused(dns, n_layers)) {
        fused::Params prm = fused_params(fused::kModeVerify, M, w);
        for (int l = 0; l < n_layers; ++l)
            prm.layers[l] = layers[l];
        set_dense(prm, dns, n_layers);
        prm.n_layers = n_layers;
        prm.x = x;
        prm.emb = emb;
        prm.V = V;
        prm.draft = draft;
        prm.argmax = argmax;
        prm.out = out;
        return launch_fused(prm, st);
    }
    k_bf16_to_f32<<<8, 256, 0, st>>>(x, M * kH, w.h);
    FGM_CHECK_LAUNCH();
    FGM_TRY(run_stack(layers, n_layers, M, w, nullptr, st, dns));
    k_rmsnorm<<<M, 256, 0, st>>>(w.h, nullptr, w.hb);
    FGM_CHECK_LAUNCH();
    const int G = lmhead_grid(sms);
    FGM_TRY(launch_lmhead(M, emb, V, w.hb, w, G, st));
    k_argmax_final<<<1, 256, 0, st>>>(w.part_val, w.part_idx, G, M, argmax ? argmax : w.argmax, nullptr,
                                      draft, out, w.status);
    FGM_CHECK_LAUNCH();
    return FGM_OK;
}

}  // namespace
}  // namespace fgm

using namespace fgm;

extern "C" {

size_t fgm_workspace_bytes(int M, int64_t V)
{
    (void)V;
    if (M < 1 || M > kMaxM)
        return 0;
    return ws_offsets().total;
}

const char *fgm_last_error(void) { return g_err; }

int fgm_version(void) { return 100; }

int fgm_moe_layer_fwd(const fgm_layer *layer, const uint16_t *x, uint16_t *y, int M,
                      int32_t *topk_ids, float *topk_w, void *ws, size_t ws_bytes, void *stream)
{
    int sms = 0;
    FGM_TRY(check_m(M));
    FGM_TRY(check_layer(layer, 0));
    if (!x || !y || !aligned16(x) || !aligned16(y))
        return fail(FGM_ERR_INVALID_ARG, "x/y NULL or not 16-byte aligned");
    if (x == y)
        return fail(FGM_ERR_INVALID_ARG, "y may not alias x");
    FGM_TRY(check_ws(ws, ws_bytes, M, 0));
    FGM_TRY(device_ready(&sms));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Ws w = ws_carve(ws);
    if (g_path != FGM_PATH_STAGED) {
        fused::Params prm = fused_params(fused::kModeLayer, M, w);
        prm.layers[0] = *layer;
        prm.n_layers = 1;
        prm.x = x;
        prm.y = y;
        prm.ids = topk_ids;
        prm.wts = topk_w;
        return launch_fused(prm, st);
    }
    k_layer_prep<<<16, 256, 0, st>>>(x, M, w.xn, w.acc);
    FGM_CHECK_LAUNCH();
    FGM_TRY(run_layer(M, layer, w, w.acc, topk_ids, topk_w, st));
    k_f32_to_bf16<<<16, 256, 0, st>>>(w.acc, M * kH, y);
    FGM_CHECK_LAUNCH();
    return FGM_OK;
}

int fgm_moe_layer_dense_fwd(const fgm_layer *layer, const fgm_mlp *dense, const uint16_t *x, uint16_t *y, int M,
                            int32_t *topk_ids, float *topk_w, void *ws, size_t ws_bytes, void *stream)
{
    FGM_TRY(check_m(M));
    FGM_TRY(check_layer(layer, 0));
    DenseArgs dn;
    FGM_TRY(check_mlp(dense, 0, &dn));
    if (!x || !y || !aligned16(x) || !aligned16(y))
        return fail(FGM_ERR_INVALID_ARG, "x/y NULL or not 16-byte aligned");
    if (x == y)
        return fail(FGM_ERR_INVALID_ARG, "y may not alias x");
    FGM_TRY(check_ws(ws, ws_bytes, M, 0));
    FGM_TRY(device_ready(nullptr));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Ws w = ws_carve(ws);
    if (g_path != FGM_PATH_STAGED && dn.parts == kMaxDense) {
        // the persistent kernel with the MLP's three parts as its always-on slots
        fused::Params prm = fused_params(fused::kModeLayer, M, w);
        prm.layers[0] = *layer;
        prm.n_layers = 1;
        prm.x = x;
        prm.y = y;
        prm.ids = topk_ids;
        prm.wts = topk_w;
        prm.dense[0] = dn;
        prm.dense_parts = kMaxDense;
        return launch_fused(prm, st);
    }
    k_layer_prep<<<16, 256, 0, st>>>(x, M, w.xn, w.acc);
    FGM_CHECK_LAUNCH();
    FGM_TRY(run_layer(M, layer, w, w.acc, topk_ids, topk_w, st, dn));
    k_f32_to_bf16<<<16, 256, 0, st>>>(w.acc, M * kH, y);
    FGM_CHECK_LAUNCH();
    return FGM_OK;
}

namespace fgm {
namespace {

int stack_impl(const fgm_layer *layers, int n_layers, const uint16_t *x, uint16_t *y, int M, int32_t *ids_trace,
               void *ws, size_t ws_bytes, void *stream, const DenseArgs *dns)
{
    int sms = 0;
    if (!x || !y || !aligned16(x) || !aligned16(y))
        return fail(FGM_ERR_INVALID_ARG, "x/y NULL or not 16-byte aligned");
    FGM_TRY(check_ws(ws, ws_bytes, M, 0));
    FGM_TRY(device_ready(&sms));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Ws w = ws_carve(ws);
    if (g_path != FGM_PATH_STAGED && dense_fused(dns, n_layers)) {
        fused::Params prm = fused_params(fused::kModeStack, M, w);
        for (int l = 0; l < n_layers; ++l)
            prm.layers[l] = layers[l];
        set_dense(prm, dns, n_layers);
        prm.n_layers = n_layers;
        prm.x = x;
        prm.y = y;
        prm.ids = ids_trace;
        return launch_fused(prm, st);
    }
    k_bf16_to_f32<<<8, 256, 0, st>>>(x, M * kH, w.h);
    FGM_CHECK_LAUNCH();
    FGM_TRY(run_stack(layers, n_layers, M, w, ids_trace, st, dns));
    k_f32_to_bf16<<<16, 256, 0, st>>>(w.h, M * kH, y);
    FGM_CHECK_LAUNCH();
    return FGM_OK;
}

int check_mlps(const fgm_mlp *mlps, int n_layers, DenseArgs *out)
{
    if (!mlps)
        return fail(FGM_ERR_INVALID_ARG, "mlps is NULL");
    for (int l = 0; l < n_layers; ++l)
        FGM_TRY(check_mlp(&mlps[l], l, &out[l]));
    return FGM_OK;
}

}  // namespace
}  // namespace fgm

int fgm_moe_stack_fwd(const fgm_layer *layers, int n_layers, const uint16_t *x, uint16_t *y, int M,
                      int32_t *ids_trace, void *ws, size_t ws_bytes, void *stream)
{
    FGM_TRY(check_m(M));
    FGM_TRY(check_layers(layers, n_layers));
    return stack_impl(layers, n_layers, x, y, M, ids_trace, ws, ws_bytes, stream, nullptr);
}

int fgm_moe_stack_dense_fwd(const fgm_layer *layers, const fgm_mlp *mlps, int n_layers, const uint16_t *x,
                            uint16_t *y, int M, int32_t *ids_trace, void *ws, size_t ws_bytes, void *stream)
{
    FGM_TRY(check_m(M));
    FGM_TRY(check_layers(layers, n_layers));
    DenseArgs dns[FGM_MAX_LAYERS];
    FGM_TRY(check_mlps(mlps, n_layers, dns));
    return stack_impl(layers, n_layers, x, y, M, ids_trace, ws, ws_bytes, stream, dns);
}

int fgm_lm_head_argmax(const uint16_t *emb, int64_t V, const uint16_t *h, int M, int32_t *argmax,
                       float *maxlogit, void *ws, size_t ws_bytes, void *stream)
{
    int sms = 0;
    FGM_TRY(check_m(M));
    FGM_TRY(check_vocab(emb, V));
    if (!h || !aligned16(h) || !argmax)
        return fail(FGM_ERR_INVALID_ARG, "h/argmax NULL or h not 16-byte aligned");
    FGM_TRY(check_ws(ws, ws_bytes, M, V));
    FGM_TRY(device_ready(&sms));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Ws w = ws_carve(ws);
    if (g_path != FGM_PATH_STAGED) {
        fused::Params prm = fused_params(fused::kModeLmHead, M, w);
        prm.x = h;
        prm.emb = emb;
        prm.V = V;
        prm.argmax = argmax;
        prm.maxlogit = maxlogit;
        return launch_fused(prm, st);
    }
    const int G = lmhead_grid(sms);
    FGM_TRY(launch_lmhead(M, emb, V, h, w, G, st));
    k_argmax_final<<<1, 256, 0, st>>>(w.part_val, w.part_idx, G, M, argmax, maxlogit, nullptr, nullptr,
                                      w.status);
    FGM_CHECK_LAUNCH();
    return FGM_OK;
}

int fgm_lm_head_argmax_fp8(const uint8_t *emb_q, const float *emb_s, int64_t V, const uint16_t *h, int M,
                           int32_t *argmax, float *maxlogit, void *ws, size_t ws_bytes, void *stream)
{
    int sms = 0;
    FGM_TRY(check_m(M));
    FGM_TRY(check_vocab_fp8(emb_q, emb_s, V));
    if (!h || !aligned16(h) || !argmax)
        return fail(FGM_ERR_INVALID_ARG, "h/argmax NULL or h not 16-byte aligned");
    FGM_TRY(check_ws(ws, ws_bytes, M, V));
    FGM_TRY(device_ready(&sms));
    return run_lmhead_fp8(emb_q, emb_s, V, h, false, M, argmax, maxlogit, nullptr, nullptr, ws_carve(ws), sms,
                          static_cast<cudaStream_t>(stream));
}

int fgm_verify_step_fp8_head(const fgm_layer *layers, int n_layers, const uint8_t *emb_q, const float *emb_s,
                             int64_t V, const uint16_t *x, const int32_t *draft, int M, int32_t *argmax,
                             int32_t *out, void *ws, size_t ws_bytes, void *stream)
{
    int sms = 0;
    FGM_TRY(check_m(M));
    FGM_TRY(check_layers(layers, n_layers));
    FGM_TRY(check_vocab_fp8(emb_q, emb_s, V));
    if (!x || !aligned16(x) || !out || (M > 1 && !draft))
        return fail(FGM_ERR_INVALID_ARG, "x/out NULL, x misaligned, or draft NULL with M > 1");
    FGM_TRY(check_ws(ws, ws_bytes, M, V));
    FGM_TRY(device_ready(&sms));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Ws w = ws_carve(ws);
    // the stack leaves the final fp32 residual stream in w.h
    if (g_path != FGM_PATH_STAGED) {
        fused::Params prm = fused_params(fused::kModeStack, M, w);
        for (int l = 0; l < n_layers; ++l)
            prm.layers[l] = layers[l];
        prm.n_layers = n_layers;
        prm.x = x;
        prm.y = w.hb;   // bf16 copy of h (unused: the lm_head kernel normalises w.h itself)
        FGM_TRY(launch_fused(prm, st));
    } else {
        k_bf16_to_f32<<<8, 256, 0, st>>>(x, M * kH, w.h);
        FGM_CHECK_LAUNCH();
        FGM_TRY(run_stack(layers, n_layers, M, w, nullptr, st));
    }
    return run_lmhead_fp8(emb_q, emb_s, V, w.h, true, M, argmax ? argmax : w.argmax, nullptr, draft, out, w, sms,
                          st);
}

int fgm_spec_verify(const int32_t *target, const int32_t *draft, int M, int32_t *out, void *stream)
{
    FGM_TRY(check_m(M));
    if (!target || !out || (M > 1 && !draft))
        return fail(FGM_ERR_INVALID_ARG, "target/out NULL, or draft NULL with M > 1");
    FGM_TRY(device_ready(nullptr));
    k_spec_verify<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(target, draft, M, out);
    FGM_CHECK_LAUNCH();
    return FGM_OK;
}

int fgm_verify_step(const fgm_layer *layers, int n_layers, const uint16_t *emb, int64_t V,
                    const uint16_t *x, const int32_t *draft, int M, int32_t *argmax, int32_t *out,
                    void *ws, size_t ws_bytes, void *stream)
{
    int sms = 0;
    FGM_TRY(check_m(M));
    FGM_TRY(check_layers(layers, n_layers));
    FGM_TRY(check_vocab(emb, V));
    if (!x || !aligned16(x) || !out || (M > 1 && !draft))
        return fail(FGM_ERR_INVALID_ARG, "x/out NULL, x misaligned, or draft NULL with M > 1");
    FGM_TRY(check_ws(ws, ws_bytes, M, V));
    FGM_TRY(device_ready(&sms));
    return verify_step_impl(layers, n_layers, emb, V, x, draft, M, argmax, out, ws,
                            static_cast<cudaStream_t>(stream), sms);
}

int fgm_verify_step_dense(const fgm_layer *layers, const fgm_mlp *mlps, int n_layers, const uint16_t *emb,
                          int64_t V, const uint16_t *x, const int32_t *draft, int M, int32_t *argmax, int32_t *out,
                          void *ws, size_t ws_bytes, void *stream)
{
    int sms = 0;
    FGM_TRY(check_m(M));
    FGM_TRY(check_layers(layers, n_layers));
    DenseArgs dns[FGM_MAX_LAYERS];
    FGM_TRY(check_mlps(mlps, n_layers, dns));
    FGM_TRY(check_vocab(emb, V));
    if (!x || !aligned16(x) || !out || (M > 1 && !draft))
        return fail(FGM_ERR_INVALID_ARG, "x/out NULL, x misaligned, or draft NULL with M > 1");
    FGM_TRY(check_ws(ws, ws_bytes, M, V));
    FGM_TRY(device_ready(&sms));
    return verify_step_impl(layers, n_layers, emb, V, x, draft, M, argmax, out, ws,
                            static_cast<cudaStream_t>(stream), sms, dns);
}

namespace fgm {
namespace {

int check_sample_args(int M, float T, const int32_t *draft, const float *u_acc, const float *u_next, float *z,
                      int32_t *out)
{
    if (!(T > 0.0f) || !std::isfinite(T) || !std::isfinite(1.0f / T))
        return fail(FGM_ERR_INVALID_ARG, "temperature T = %g: needs a finite T > 0 with 1/T finite", (double)T);
    if (!u_next || !z || !out || (M > 1 && (!draft || !u_acc)))
        return fail(FGM_ERR_INVALID_ARG, "u_next/z/out NULL, or draft/u_acc NULL with M > 1");
    if ((reinterpret_cast<uintptr_t>(z) | reinterpret_cast<uintptr_t>(u_next) |
         reinterpret_cast<uintptr_t>(u_acc)) & 3u)
        return fail(FGM_ERR_INVALID_ARG, "z/u_next/u_acc not 4-byte aligned");
    return FGM_OK;
}

void set_sample(fused::Params &prm, float T, const int32_t *draft, const float *u_acc, const float *u_next,
                float *z, int32_t *argmax, int32_t *out, const Ws &w)
{
    prm.z = z;
    prm.inv_t = 1.0f / T;
    prm.draft = draft;
    prm.u_acc = u_acc;
    prm.u_next = u_next;
    prm.argmax = argmax ? argmax : w.argmax;
    prm.out = out;
}

}  // namespace
}  // namespace fgm

int fgm_lm_head_sample(const uint16_t *emb, int64_t V, const uint16_t *h, int M, float T, const int32_t *draft,
                       const float *u_acc, const float *u_next, float *z, int32_t *argmax, int32_t *out,
                       void *ws, size_t ws_bytes, void *stream)
{
    FGM_TRY(check_m(M));
    FGM_TRY(check_vocab(emb, V));
    if (!h || !aligned16(h))
        return fail(FGM_ERR_INVALID_ARG, "h NULL or not 16-byte aligned");
    FGM_TRY(check_sample_args(M, T, draft, u_acc, u_next, z, out));
    FGM_TRY(check_ws(ws, ws_bytes, M, V));
    FGM_TRY(device_ready(nullptr));
    Ws w = ws_carve(ws);
    fused::Params prm = fused_params(fused::kModeLmHead, M, w);
    prm.x = h;
    prm.emb = emb;
    prm.V = V;
    set_sample(prm, T, draft, u_acc, u_next, z, argmax, out, w);
    return launch_fused(prm, static_cast<cudaStream_t>(stream));
}

int fgm_verify_step_sample(const fgm_layer *layers, int n_layers, const uint16_t *emb, int64_t V,
                           const uint16_t *x, const int32_t *draft, int M, float T, const float *u_acc,
                           const float *u_next, float *z, int32_t *argmax, int32_t *out, void *ws,
                           size_t ws_bytes, void *stream)
{
    FGM_TRY(check_m(M));
    FGM_TRY(check_layers(layers, n_layers));
    FGM_TRY(check_vocab(emb, V));
    if (!x || !aligned16(x))
        return fail(FGM_ERR_INVALID_ARG, "x NULL or not 16-byte aligned");
    FGM_TRY(check_sample_args(M, T, draft, u_acc, u_next, z, out));
    FGM_TRY(check_ws(ws, ws_bytes, M, V));
    FGM_TRY(device_ready(nullptr));
    Ws w = ws_carve(ws);
    fused::Params prm = fused_params(fused::kModeVerify, M, w);
    for (int l = 0; l < n_layers; ++l)
        prm.layers[l] = layers[l];
    prm.n_layers = n_layers;
    prm.x = x;
    prm.emb = emb;
    prm.V = V;
    set_sample(prm, T, draft, u_acc, u_next, z, argmax, out, w);
    return launch_fused(prm, static_cast<cudaStream_t>(stream));
}

int fgm_verify_step_host(const fgm_layer *layers, int n_layers, const uint16_t *emb, int64_t V,
                         const uint16_t *x_host, const int32_t *draft_host, int M, int32_t *out_host,
                         void *ws, size_t ws_bytes, void *stream)
{
    int sms = 0;
    FGM_TRY(check_m(M));
    FGM_TRY(check_layers(layers, n_layers));
    FGM_TRY(check_vocab(emb, V));
    if (!x_host || !out_host || (M > 1 && !draft_host))
        return fail(FGM_ERR_INVALID_ARG, "x_host/out_host NULL, or draft_host NULL with M > 1");
    FGM_TRY(check_ws(ws, ws_bytes, M, V));
    FGM_TRY(device_ready(&sms));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Ws w = ws_carve(ws);
    FGM_CUDA(cudaMemcpyAsync(w.io_x, x_host, sizeof(uint16_t) * M * kH, cudaMemcpyHostToDevice, st));
    if (M > 1)
        FGM_CUDA(cudaMemcpyAsync(w.io_draft, draft_host, sizeof(int32_t) * (M - 1), cudaMemcpyHostToDevice, st));
    FGM_TRY(verify_step_impl(layers, n_layers, emb, V, w.io_x, w.io_draft, M, nullptr, w.io_out, ws, st, sms));
    FGM_CUDA(cudaMemcpyAsync(out_host, w.io_out, sizeof(int32_t) * 2, cudaMemcpyDeviceToHost, st));
    FGM_CUDA(cudaStreamSynchronize(st));
    return FGM_OK;
}

int fgm_select_path(int path)
{
    const int prev = g_path;
    if (path == FGM_PATH_FUSED || path == FGM_PATH_STAGED || path == FGM_PATH_FUSED_TC || path == FGM_PATH_FUSED_MMA)
        g_path = path;
    return prev;
}

int fgm_debug_stall_next_launch(void)
{
    g_debug_stall = 1;
    return FGM_OK;
}

int fgm_debug_stall_next_launch_at(int layer)
{
    if (layer < 0 || layer >= FGM_MAX_LAYERS)
        return fail(FGM_ERR_INVALID_ARG, "layer %d outside [0, %d)", layer, FGM_MAX_LAYERS);
    g_debug_stall = layer + 1;
    return FGM_OK;
}

int fgm_set_phase_trace(long long *buf, size_t n)
{
    g_trace = buf;
    g_trace_n = buf ? n : 0;
    return FGM_OK;
}

long long fgm_set_wait_limit_ns(long long ns)
{
    const long long prev = g_timeout_ns;
    if (ns >= 0)
        g_timeout_ns = ns;
    return prev;
}

int fgm_read_wait_report(void *ws, size_t ws_bytes, int32_t *report, void *stream)
{
    FGM_TRY(check_ws(ws, ws_bytes, 1, 0));
    if (!report)
        return fail(FGM_ERR_INVALID_ARG, "report is NULL");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Ws w = ws_carve(ws);
    FGM_CUDA(cudaMemcpyAsync(report, w.status + 1, 4 * sizeof(int32_t), cudaMemcpyDeviceToHost, st));
    FGM_CUDA(cudaStreamSynchronize(st));
    return FGM_OK;
}

int fgm_workspace_init(void *ws, size_t ws_bytes, void *stream)
{
    FGM_TRY(check_ws(ws, ws_bytes, 1, 0));
    FGM_CUDA(cudaMemsetAsync(ws, 0, ws_offsets().total, static_cast<cudaStream_t>(stream)));
    return FGM_OK;
}

int fgm_read_status(void *ws, size_t ws_bytes, int clear, int32_t *status, void *stream)
{
    FGM_TRY(check_ws(ws, ws_bytes, 1, 0));
    if (!status)
        return fail(FGM_ERR_INVALID_ARG, "status is NULL");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Ws w = ws_carve(ws);
    FGM_CUDA(cudaMemcpyAsync(status, w.status, sizeof(int32_t), cudaMemcpyDeviceToHost, st));
    FGM_CUDA(cudaStreamSynchronize(st));
    if (clear)
        FGM_CUDA(cudaMemsetAsync(w.status, 0, sizeof(int32_t), st));
    return FGM_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- allocation-free layer call
//
// fgm_moe_layer_fwd_noalloc runs fgm_moe_layer_fwd on scratch that the library
// owns: a module-scope device array reserved when the CUDA module is loaded,
// so the call itself never allocates. Its capacity is one full workspace
// (M <= FGM_MAX_M = 8, V = 0); the array is shared by every caller on a device.

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // >= fgm_workspace_bytes(8, 0)

}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

void *g_noalloc_base[kMaxDevices];  // device address of g_noalloc_scratch, per device
std::mutex g_noalloc_mu;

// Resolves (once per device, with that device current) the address of the
// module-scope scratch. Nothing is allocated; the CUDA runtime may load the
// module on this first query.
int noalloc_scratch(void **base)
{
    int dev = 0;
    FGM_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices)
        return fail(FGM_ERR_DEVICE, "device index %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_base[dev]) {
        if (ws_offsets().total > kNoAllocScratchBytes)
            return fail(FGM_ERR_WORKSPACE, "built-in scratch of %zu bytes is below the %zu a layer call needs",
                        kNoAllocScratchBytes, ws_offsets().total);
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p)
            return fail(FGM_ERR_CUDA, "cudaGetSymbolAddress(built-in scratch) failed: %s",
                        cudaGetErrorString(e));
        if (reinterpret_cast<uintptr_t>(p) & 255u)
            return fail(FGM_ERR_WORKSPACE, "built-in scratch is not 256-byte aligned");
        g_noalloc_base[dev] = p;
    }
    *base = g_noalloc_base[dev];
    return FGM_OK;
}

}  // namespace

extern "C" int fgm_moe_layer_fwd_noalloc(const fgm_layer *layer, const uint16_t *x, uint16_t *y, int M,
                                         int32_t *topk_ids, float *topk_w, void *stream)
{
    if (M < 1 || M > kMaxM)
        return fail(FGM_ERR_INVALID_ARG,
                    "M = %d outside [1, %d]: the built-in scratch of fgm_moe_layer_fwd_noalloc holds at most "
                    "%d tokens", M, kMaxM, kMaxM);
    FGM_TRY(check_layer(layer, 0));
    if (!x || !y || !aligned16(x) || !aligned16(y))
        return fail(FGM_ERR_INVALID_ARG, "x/y NULL or not 16-byte aligned");
    if (x == y)
        return fail(FGM_ERR_INVALID_ARG, "y may not alias x");
    FGM_TRY(device_ready(nullptr));
    void *base = nullptr;
    FGM_TRY(noalloc_scratch(&base));
    // The status word and the grid-barrier counters must start at zero; the
    // kernels initialise every other region they read.
    const WsOffsets o = ws_offsets();
    FGM_CUDA(cudaMemsetAsync(static_cast<char *>(base) + o.status, 0, o.xterms - o.status,
                             static_cast<cudaStream_t>(stream)));
    return fgm_moe_layer_fwd(layer, x, y, M, topk_ids, topk_w, base, o.total, stream);
}
