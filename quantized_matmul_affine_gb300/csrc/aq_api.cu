// C ABI of libaq: argument checks, the dispatch rule, counters, host I/O.
//
// The interface follows affineSplitMma on the mlx-bun pages (@mlx-bun/inference
// 1.0.0, kernels/quantization/affine-split-mma.ts): x with any number of rows
// times W^T, y in x's dtype, an error for no rows; plus the pack step and the
// explicit-variant and host-memory entry points described in aq.h.
#include "aq_internal.h"

#include <cudaTypedefs.h>

#include <atomic>
#include <cstdio>
#include <mutex>
#include <cstdlib>
#include <cstring>

namespace aq {

namespace {

std::atomic<uint64_t> g_calls[AQ_NUM_VARIANTS];
std::atomic<int> g_sms_cache[64];

// Largest M that the streaming small-M kernel takes under the automatic rule
// when the resident kernel does not apply: past 16 rows the tensor-core
// kernel measured faster on GB300.  AQ_QMV_MAX_M overrides it for
// experiments.
int qmv_max_m() {
    static const int v = [] {
        const char *e = std::getenv("AQ_QMV_MAX_M");
        if (e && *e) return std::atoi(e);
        return 16;
    }();
    return v;
}

}  // namespace

#ifdef AQ_TEST_HOOKS
int g_test_withhold = 0;
int g_test_cluster_split = 0;
#endif

int num_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return 152;
    }
    int v = g_sms_cache[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
        cudaGetLastError();
        return 152;
    }
    g_sms_cache[dev].store(v, std::memory_order_relaxed);
    return v;
}

bool tmap_encode(CUtensorMap *tm, CUtensorMapDataType type, int rank, const void *base,
                 const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box,
                 CUtensorMapSwizzle swizzle) {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        else
            cudaGetLastError();
    });
    if (!fn || rank < 1 || rank > 5) return false;
    cuuint64_t d[5], st[4];
    cuuint32_t bx[5], es[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = (cuuint64_t)dims[i];
        bx[i] = (cuuint32_t)box[i];
        es[i] = 1;
        if (i + 1 < rank) st[i] = (cuuint64_t)strides_bytes[i];
    }
    return fn(tm, type, (cuuint32_t)rank, const_cast<void *>(base), d, st, bx, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Largest M that the resident small-M kernel takes under the automatic rule
// (AQ_GEMV_MAX_M overrides it for experiments): it serves up to four 8-column
// blocks, and measured faster than qmv at every M from 1 to 16 but the
// single-row case below, and 1.9-3.3x faster than tc from 17 to 32 (GB300:
// 3-bit 10240x5120 at M = 32, 20.8 against 39.4 us).
static int gemv_max_m() {
    static const int v = [] {
        const char *e = std::getenv("AQ_GEMV_MAX_M");
        if (e && *e) return std::atoi(e);
        return 32;
    }();
    return v;
}

// A single activation row goes to the resident kernel only when its CTAs
// take all their rows in one pass (N <= 128 rows x SMs); past that the
// streaming small-M kernel keeps pace or wins (measured on GB300 at 4 bits,
// M = 1: gemv is 11-29% faster on 13824x5120 and 4096x14336, within 1% on
// 5120x13824; two passes: 5% faster on 28672x8192 but 8% slower on
// 32000x4096; 128256x4096 and 57344x8192: 18-23% slower).
static bool gemv_for_m1(const MatmulArgs &a) { return a.N <= 128ll * num_sms(); }

// Past 32 activation rows the tensor-core kernel takes every shape: with
// fewer weight tiles than SMs it shares tiles among the CTAs of a cluster
// (the clustered K split), which left the swapped-role kernel (still
// available as AQ_VARIANT_TCW) behind on every shape measured (GB300, us:
// 10240x5120 3-bit at M = 33/64/128: 23.1/23.2/26.6 against 27.8/29.7/33.7;
// 4096x4096 at 64/128: 12.0/14.0 against 24.2/29.0; 5120x13824 at 64: 28.3
// against 64.0; 5120x5120 at 128: 17.3 against 39.4; 1024x5120 at 64: 9.8
// against 15.1; 13824x5120 at 128: 30.5 against 43.2).

// The dispatch rule.  Returns the variant for the arguments (alignment
// included), never AQ_VARIANT_AUTO.
static int choose(const MatmulArgs &a) {
    const bool gemv_first = a.M > 1 || gemv_for_m1(a);
    if (a.M <= gemv_max_m() && gemv_first && gemv_supported(a)) return AQ_VARIANT_GEMV;
    const bool qmv = qmv_supported(a);
    const bool tc = tc_supported(a);
    if (qmv && (a.M <= qmv_max_m() || !tc)) return AQ_VARIANT_QMV;
    if (tc) return AQ_VARIANT_TC;
    return AQ_VARIANT_GENERIC;
}

static aq_status check_args(const MatmulArgs &a) {
    if (a.M < 1 || a.N < 1 || a.K < 64 || a.K % 64 != 0) return AQ_ERR_INVALID_ARG;
    if (a.bits != 3 && a.bits != 4) return AQ_ERR_INVALID_ARG;
    if (a.dtype != AQ_F16 && a.dtype != AQ_BF16) return AQ_ERR_INVALID_ARG;
    if (!a.x || !a.Wq || !a.scales || !a.biases || !a.out) return AQ_ERR_INVALID_ARG;
    if (a.M > (int64_t)1 << 31 || a.N > (int64_t)1 << 31 || a.K > (int64_t)1 << 31)
        return AQ_ERR_UNSUPPORTED;
    if (!aligned(a.x, 2) || !aligned(a.out, 2) || !aligned(a.scales, 2) || !aligned(a.biases, 2) ||
        !aligned(a.Wq, 4))
        return AQ_ERR_MISALIGNED;
    return AQ_OK;
}

static aq_status run(int variant, const MatmulArgs &a) {
    aq_status st = check_args(a);
    if (st != AQ_OK) return st;
    if (variant == AQ_VARIANT_AUTO) variant = choose(a);
    cudaError_t err;
    switch (variant) {
        case AQ_VARIANT_GENERIC:
            if (!generic_supported(a)) return AQ_ERR_UNSUPPORTED;
            err = generic_launch(a);
            break;
        case AQ_VARIANT_QMV:
            if (!qmv_supported(a)) return AQ_ERR_UNSUPPORTED;
            err = qmv_launch(a);
            break;
        case AQ_VARIANT_TC:
            if (!tc_supported(a)) return AQ_ERR_UNSUPPORTED;
            err = tc_launch(a);
            break;
        case AQ_VARIANT_GEMV:
            if (!gemv_supported(a)) return AQ_ERR_UNSUPPORTED;
            err = gemv_launch(a);
            break;
        case AQ_VARIANT_TCW:
            if (!tcw_supported(a)) return AQ_ERR_UNSUPPORTED;
            err = tcw_launch(a);
            break;
        default:
            return AQ_ERR_INVALID_ARG;
    }
    if (err != cudaSuccess) return AQ_ERR_CUDA;
    g_calls[variant].fetch_add(1, std::memory_order_relaxed);
    return AQ_OK;
}

static MatmulArgs make_args(int dtype, const void *x, const uint32_t *Wq, const void *scales,
                            const void *biases, int64_t M, int64_t N, int64_t K, int bits,
                            void *out, void *stream) {
    MatmulArgs a;
    a.x = x;
    a.Wq = Wq;
    a.scales = scales;
    a.biases = biases;
    a.out = out;
    a.M = M;
    a.N = N;
    a.K = K;
    a.bits = bits;
    a.dtype = dtype;
    a.stream = static_cast<cudaStream_t>(stream);
    return a;
}

}  // namespace aq

using namespace aq;

extern "C" {

static bool valid_width(int bits) {
    return bits == 2 || bits == 3 || bits == 4 || bits == 5 || bits == 6 || bits == 8;
}

aq_status aq_pack(const uint8_t *codes_dev, int64_t N, int64_t K, int bits, uint32_t *words_dev,
                  void *stream) {
    if (N < 0 || K < 0 || K % 32 != 0 || !valid_width(bits)) return AQ_ERR_INVALID_ARG;
    if (N == 0 || K == 0) return AQ_OK;
    if (!codes_dev || !words_dev) return AQ_ERR_INVALID_ARG;
    if (!aligned(words_dev, 4)) return AQ_ERR_MISALIGNED;
    if (pack_launch(codes_dev, N, K, bits, words_dev, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return AQ_ERR_CUDA;
    return AQ_OK;
}

static aq_status quantize_entry(int dtype, const void *w_dev, int64_t N, int64_t K, int bits,
                                uint32_t *Wq_dev, void *scales_dev, void *biases_dev,
                                void *stream) {
    if (N < 0 || K < 0 || K % 64 != 0 || (bits != 3 && bits != 4)) return AQ_ERR_INVALID_ARG;
    if (N == 0 || K == 0) return AQ_OK;
    if (!w_dev || !Wq_dev || !scales_dev || !biases_dev) return AQ_ERR_INVALID_ARG;
    if (!aligned(w_dev, 16) || !aligned(Wq_dev, 4) || !aligned(scales_dev, 2) ||
        !aligned(biases_dev, 2))
        return AQ_ERR_MISALIGNED;
    if (quantize_launch(dtype, w_dev, N, K, bits, Wq_dev, scales_dev, biases_dev,
                        static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return AQ_ERR_CUDA;
    return AQ_OK;
}

aq_status aq_quantize_ex(int dtype, const void *w_dev, int64_t N, int64_t K, int bits,
                         int group_size, uint32_t *Wq_dev, void *scales_dev, void *biases_dev,
                         void *stream) {
    if (dtype != AQ_F16 && dtype != AQ_BF16) return AQ_ERR_INVALID_ARG;
    if (bits == 3 || bits == 4)
        if (group_size == 64)
            return quantize_entry(dtype, w_dev, N, K, bits, Wq_dev, scales_dev, biases_dev, stream);
    if (group_size != 32 && group_size != 64 && group_size != 128) return AQ_ERR_INVALID_ARG;
    if (N < 0 || K < 0 || K % group_size != 0 || !valid_width(bits)) return AQ_ERR_INVALID_ARG;
    if (N == 0 || K == 0) return AQ_OK;
    if (!w_dev || !Wq_dev || !scales_dev || !biases_dev) return AQ_ERR_INVALID_ARG;
    if (!aligned(w_dev, 2) || !aligned(Wq_dev, 4) || !aligned(scales_dev, 2) ||
        !aligned(biases_dev, 2))
        return AQ_ERR_MISALIGNED;
    if (quantize_launch_g(dtype, w_dev, N, K, bits, group_size, Wq_dev, scales_dev, biases_dev,
                          static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return AQ_ERR_CUDA;
    return AQ_OK;
}

aq_status aq_quantize(const void *w_dev, int64_t N, int64_t K, int bits, uint32_t *Wq_dev,
                      void *scales_dev, void *biases_dev, void *stream) {
    return quantize_entry(AQ_F16, w_dev, N, K, bits, Wq_dev, scales_dev, biases_dev, stream);
}

aq_status aq_quantize_bf16(const void *w_dev, int64_t N, int64_t K, int bits, uint32_t *Wq_dev,
                           void *scales_dev, void *biases_dev, void *stream) {
    return quantize_entry(AQ_BF16, w_dev, N, K, bits, Wq_dev, scales_dev, biases_dev, stream);
}

aq_status aq_matmul(const void *x_dev, const uint32_t *Wq_dev, const void *scales_dev,
                    const void *biases_dev, int64_t M, int64_t N, int64_t K, int bits,
                    void *out_dev, void *stream) {
    return run(AQ_VARIANT_AUTO, make_args(AQ_F16, x_dev, Wq_dev, scales_dev, biases_dev, M, N, K,
                                          bits, out_dev, stream));
}

aq_status aq_matmul_bf16(const void *x_dev, const uint32_t *Wq_dev, const void *scales_dev,
                         const void *biases_dev, int64_t M, int64_t N, int64_t K, int bits,
                         void *out_dev, void *stream) {
    return run(AQ_VARIANT_AUTO, make_args(AQ_BF16, x_dev, Wq_dev, scales_dev, biases_dev, M, N, K,
                                          bits, out_dev, stream));
}

aq_status aq_matmul_ex(int dtype, const void *x_dev, const uint32_t *Wq_dev,
                       const void *scales_dev, const void *biases_dev, int64_t M, int64_t N,
                       int64_t K, int bits, int group_size, void *out_dev, void *stream) {
    if (dtype != AQ_F16 && dtype != AQ_BF16) return AQ_ERR_INVALID_ARG;
    MatmulArgs a = make_args(dtype, x_dev, Wq_dev, scales_dev, biases_dev, M, N, K, bits, out_dev,
                             stream);
    if ((bits == 3 || bits == 4) && group_size == 64) return run(AQ_VARIANT_AUTO, a);
    if (group_size != 32 && group_size != 64 && group_size != 128) return AQ_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < group_size || K % group_size != 0 || !valid_width(bits))
        return AQ_ERR_INVALID_ARG;
    if (!x_dev || !Wq_dev || !scales_dev || !biases_dev || !out_dev) return AQ_ERR_INVALID_ARG;
    if (!aligned(x_dev, 2) || !aligned(Wq_dev, 4) || !aligned(scales_dev, 2) ||
        !aligned(biases_dev, 2) || !aligned(out_dev, 2))
        return AQ_ERR_MISALIGNED;
    if (!generic_supported_g(a, group_size)) return AQ_ERR_UNSUPPORTED;
    // Past 4 rows the tensor-core kernel with the general-width
    // dequantisation, where its shape and alignment rules hold (measured at
    // 4096 x 4096, 8 bits: 20.8 us at 4 to 16 rows against 19.3 / 33.2 /
    // 56.5 us on the segment kernel at 4 / 8 / 16 rows, which re-reads the
    // staged x per output row); otherwise up to 32 rows the segment kernel;
    // else the plain kernel.
    int variant;
    cudaError_t e;
    if (M > 4 && tc_supported_g(a, group_size)) {
        variant = AQ_VARIANT_TC;
        e = tc_launch_g(a, group_size);
    } else {
        variant = AQ_VARIANT_GENERIC;
        e = segv_supported(a, group_size) ? segv_launch(a, group_size)
                                          : generic_launch_g(a, group_size);
    }
    if (e != cudaSuccess) return AQ_ERR_CUDA;
    g_calls[variant].fetch_add(1, std::memory_order_relaxed);
    return AQ_OK;
}

aq_status aq_attention_decode(int dtype, const void *q_dev, const uint32_t *k_words_dev,
                              const void *k_scales_dev, const void *k_biases_dev,
                              const uint32_t *v_words_dev, const void *v_scales_dev,
                              const void *v_biases_dev, int64_t H, int64_t KV, int64_t N,
                              int64_t D, int bits, int group_size, void *out_dev, void *stream) {
    if (dtype != AQ_F16 && dtype != AQ_BF16) return AQ_ERR_INVALID_ARG;
    if (!q_dev || !k_words_dev || !k_scales_dev || !k_biases_dev || !v_words_dev ||
        !v_scales_dev || !v_biases_dev || !out_dev)
        return AQ_ERR_INVALID_ARG;
    if (H < 1 || KV < 1 || N < 1 || D < 1 || H % KV != 0) return AQ_ERR_INVALID_ARG;
    if ((bits != 4 && bits != 8) ||
        (group_size != 32 && group_size != 64 && group_size != 128) || D % group_size != 0)
        return AQ_ERR_INVALID_ARG;
    if (!aligned(q_dev, 2) || !aligned(out_dev, 2) || !aligned(k_words_dev, 16) ||
        !aligned(v_words_dev, 16) || !aligned(k_scales_dev, 16) || !aligned(k_biases_dev, 16) ||
        !aligned(v_scales_dev, 16) || !aligned(v_biases_dev, 16))
        return AQ_ERR_MISALIGNED;
    if (!attention_supported(H, KV, N, D, bits, group_size)) return AQ_ERR_UNSUPPORTED;
    if (attention_launch(dtype, q_dev, k_words_dev, k_scales_dev, k_biases_dev, v_words_dev,
                         v_scales_dev, v_biases_dev, H, KV, N, D, bits, group_size, out_dev,
                         nullptr, 0, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return AQ_ERR_CUDA;
    return AQ_OK;
}

aq_status aq_attention_decode_static(int dtype, const void *q_dev, const uint32_t *k_words_dev,
                                     const void *k_scales_dev, const void *k_biases_dev,
                                     const uint32_t *v_words_dev, const void *v_scales_dev,
                                     const void *v_biases_dev, int64_t H, int64_t KV, int64_t N,
                                     int64_t D, int bits, int group_size, void *out_dev,
                                     void *stream) {
    if (dtype != AQ_F16 && dtype != AQ_BF16) return AQ_ERR_INVALID_ARG;
    if (!q_dev || !k_words_dev || !k_scales_dev || !k_biases_dev || !v_words_dev ||
        !v_scales_dev || !v_biases_dev || !out_dev)
        return AQ_ERR_INVALID_ARG;
    if (H < 1 || KV < 1 || N < 1 || D < 1 || H % KV != 0) return AQ_ERR_INVALID_ARG;
    if ((bits != 4 && bits != 8) ||
        (group_size != 32 && group_size != 64 && group_size != 128) || D % group_size != 0)
        return AQ_ERR_INVALID_ARG;
    if (!aligned(q_dev, 2) || !aligned(out_dev, 2) || !aligned(k_words_dev, 16) ||
        !aligned(v_words_dev, 16) || !aligned(k_scales_dev, 16) || !aligned(k_biases_dev, 16) ||
        !aligned(v_scales_dev, 16) || !aligned(v_biases_dev, 16))
        return AQ_ERR_MISALIGNED;
    if (!attention_supported(H, KV, N, D, bits, group_size)) return AQ_ERR_UNSUPPORTED;
    // the plan aq_attention_decode_ws takes with a workspace of the size it
    // asks for; refused (nothing queued) when that is larger than the scratch
    const size_t need = attention_workspace_bytes(H, KV, N, D, bits, group_size);
    if (need > (size_t)AQ_ATTENTION_STATIC_SCRATCH_BYTES) return AQ_ERR_UNSUPPORTED;
    void *scratch = need > 0 ? attention_static_scratch() : nullptr;
    if (need > 0 && !scratch) return AQ_ERR_CUDA;
    if (attention_launch(dtype, q_dev, k_words_dev, k_scales_dev, k_biases_dev, v_words_dev,
                         v_scales_dev, v_biases_dev, H, KV, N, D, bits, group_size, out_dev,
                         scratch, need, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return AQ_ERR_CUDA;
    return AQ_OK;
}

size_t aq_attention_workspace_bytes(int64_t H, int64_t KV, int64_t N, int64_t D, int bits,
                                    int group_size) {
    if (H < 1 || KV < 1 || N < 1 || H % KV != 0) return 0;
    if (!attention_supported(H, KV, N, D, bits, group_size)) return 0;
    return attention_workspace_bytes(H, KV, N, D, bits, group_size);
}

aq_status aq_attention_decode_ws(int dtype, const void *q_dev, const uint32_t *k_words_dev,
                                 const void *k_scales_dev, const void *k_biases_dev,
                                 const uint32_t *v_words_dev, const void *v_scales_dev,
                                 const void *v_biases_dev, int64_t H, int64_t KV, int64_t N,
                                 int64_t D, int bits, int group_size, void *out_dev,
                                 void *workspace_dev, size_t workspace_bytes, void *stream) {
    if (dtype != AQ_F16 && dtype != AQ_BF16) return AQ_ERR_INVALID_ARG;
    if (!q_dev || !k_words_dev || !k_scales_dev || !k_biases_dev || !v_words_dev ||
        !v_scales_dev || !v_biases_dev || !out_dev || (workspace_bytes > 0 && !workspace_dev))
        return AQ_ERR_INVALID_ARG;
    if (H < 1 || KV < 1 || N < 1 || D < 1 || H % KV != 0) return AQ_ERR_INVALID_ARG;
    if ((bits != 4 && bits != 8) ||
        (group_size != 32 && group_size != 64 && group_size != 128) || D % group_size != 0)
        return AQ_ERR_INVALID_ARG;
    if (!aligned(q_dev, 2) || !aligned(out_dev, 2) || !aligned(k_words_dev, 16) ||
        !aligned(v_words_dev, 16) || !aligned(k_scales_dev, 16) || !aligned(k_biases_dev, 16) ||
        !aligned(v_scales_dev, 16) || !aligned(v_biases_dev, 16) ||
        !aligned(workspace_dev, 256))
        return AQ_ERR_MISALIGNED;
    if (!attention_supported(H, KV, N, D, bits, group_size)) return AQ_ERR_UNSUPPORTED;
    if (attention_launch(dtype, q_dev, k_words_dev, k_scales_dev, k_biases_dev, v_words_dev,
                         v_scales_dev, v_biases_dev, H, KV, N, D, bits, group_size, out_dev,
                         workspace_bytes > 0 ? workspace_dev : nullptr, workspace_bytes,
                         static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return AQ_ERR_CUDA;
    return AQ_OK;
}

aq_status aq_matmul_multi(int dtype, const void *x_dev, int nproj, const uint32_t *const *Wq_dev,
                          const void *const *scales_dev, const void *const *biases_dev,
                          const int64_t *N, int64_t M, int64_t K, int bits, void *const *out_dev,
                          void *stream) {
    if (dtype != AQ_F16 && dtype != AQ_BF16) return AQ_ERR_INVALID_ARG;
    if (nproj < 1 || nproj > AQ_MAX_PROJ || !Wq_dev || !scales_dev || !biases_dev || !N ||
        !out_dev)
        return AQ_ERR_INVALID_ARG;
    MultiArgs m{};
    m.a = make_args(dtype, x_dev, nullptr, nullptr, nullptr, M, 0, K, bits, nullptr, stream);
    m.nproj = nproj;
    m.gate_up = false;
    MatmulArgs each[AQ_MAX_PROJ];
    for (int j = 0; j < nproj; ++j) {
        each[j] = make_args(dtype, x_dev, Wq_dev[j], scales_dev[j], biases_dev[j], M, N[j], K,
                            bits, out_dev[j], stream);
        const aq_status st = check_args(each[j]);
        if (st != AQ_OK) return st;
        m.Wq[j] = Wq_dev[j];
        m.scales[j] = scales_dev[j];
        m.biases[j] = biases_dev[j];
        m.out[j] = out_dev[j];
        m.N[j] = N[j];
    }
    if (M <= gemv_max_m() && gemv_multi_supported(m)) {
        if (gemv_launch_multi(m) != cudaSuccess) return AQ_ERR_CUDA;
        g_calls[AQ_VARIANT_GEMV].fetch_add(1, std::memory_order_relaxed);
        return AQ_OK;
    }
    // otherwise one launch per projection, each by the dispatch rule
    for (int j = 0; j < nproj; ++j) {
        const aq_status st = run(AQ_VARIANT_AUTO, each[j]);
        if (st != AQ_OK) return st;
    }
    return AQ_OK;
}

aq_status aq_matmul_gate_up(int dtype, const void *x_dev, const uint32_t *Wg_dev,
                            const void *scales_g_dev, const void *biases_g_dev,
                            const uint32_t *Wu_dev, const void *scales_u_dev,
                            const void *biases_u_dev, int64_t M, int64_t N, int64_t K, int bits,
                            void *out_dev, void *stream) {
    if (dtype != AQ_F16 && dtype != AQ_BF16) return AQ_ERR_INVALID_ARG;
    const MatmulArgs g = make_args(dtype, x_dev, Wg_dev, scales_g_dev, biases_g_dev, M, N, K,
                                   bits, out_dev, stream);
    const MatmulArgs u = make_args(dtype, x_dev, Wu_dev, scales_u_dev, biases_u_dev, M, N, K,
                                   bits, out_dev, stream);
    aq_status st = check_args(g);
    if (st == AQ_OK) st = check_args(u);
    if (st != AQ_OK) return st;
    MultiArgs m{};
    m.a = g;
    m.nproj = 2;
    m.gate_up = true;
    m.Wq[0] = Wg_dev;
    m.scales[0] = scales_g_dev;
    m.biases[0] = biases_g_dev;
    m.Wq[1] = Wu_dev;
    m.scales[1] = scales_u_dev;
    m.biases[1] = biases_u_dev;
    m.N[0] = m.N[1] = N;
    m.out[0] = m.out[1] = out_dev;
    if (!gemv_multi_supported(m)) return AQ_ERR_UNSUPPORTED;
    if (gemv_launch_multi(m) != cudaSuccess) return AQ_ERR_CUDA;
    g_calls[AQ_VARIANT_GEMV].fetch_add(1, std::memory_order_relaxed);
    return AQ_OK;
}

aq_status aq_matmul_variant(int variant, int dtype, const void *x_dev, const uint32_t *Wq_dev,
                            const void *scales_dev, const void *biases_dev, int64_t M, int64_t N,
                            int64_t K, int bits, void *out_dev, void *stream) {
    if (variant < AQ_VARIANT_AUTO || variant >= AQ_NUM_VARIANTS) return AQ_ERR_INVALID_ARG;
    return run(variant, make_args(dtype, x_dev, Wq_dev, scales_dev, biases_dev, M, N, K, bits,
                                  out_dev, stream));
}

aq_status aq_matmul_host(int dtype, const void *x_host, const uint32_t *Wq_dev,
                         const void *scales_dev, const void *biases_dev, int64_t M, int64_t N,
                         int64_t K, int bits, void *out_host, void *x_dev, void *out_dev,
                         void *stream) {
    MatmulArgs a = make_args(dtype, x_dev, Wq_dev, scales_dev, biases_dev, M, N, K, bits,
                             out_dev, stream);
    aq_status st = check_args(a);
    if (st != AQ_OK) return st;
    if (!x_host || !out_host) return AQ_ERR_INVALID_ARG;
    const size_t xbytes = (size_t)M * (size_t)K * 2, ybytes = (size_t)M * (size_t)N * 2;
    if (cudaMemcpyAsync(x_dev, x_host, xbytes, cudaMemcpyHostToDevice, a.stream) != cudaSuccess)
        return AQ_ERR_CUDA;
    st = run(AQ_VARIANT_AUTO, a);
    if (st != AQ_OK) return st;
    if (cudaMemcpyAsync(out_host, out_dev, ybytes, cudaMemcpyDeviceToHost, a.stream) !=
        cudaSuccess)
        return AQ_ERR_CUDA;
    if (cudaStreamSynchronize(a.stream) != cudaSuccess) return AQ_ERR_CUDA;
    return AQ_OK;
}

int aq_select(int64_t M, int64_t N, int64_t K, int bits, int dtype) {
    // Placeholder addresses with 256-byte alignment: the plan only looks at
    // their alignment, never dereferences them.
    const uintptr_t fake = 0x100000;
    MatmulArgs a = make_args(dtype, (const void *)fake, (const uint32_t *)fake, (const void *)fake,
                             (const void *)fake, M, N, K, bits, (void *)fake, nullptr);
    if (check_args(a) != AQ_OK) return -1;
    return choose(a);
}

int aq_describe(int64_t M, int64_t N, int64_t K, int bits, int dtype, char *buf, int buflen) {
    if (!buf || buflen < 1) return -1;
    const uintptr_t fake = 0x100000;
    MatmulArgs a = make_args(dtype, (const void *)fake, (const uint32_t *)fake, (const void *)fake,
                             (const void *)fake, M, N, K, bits, (void *)fake, nullptr);
    if (check_args(a) != AQ_OK) return snprintf(buf, buflen, "invalid arguments");
    switch (choose(a)) {
        case AQ_VARIANT_GEMV: return gemv_describe(a, buf, buflen);
        case AQ_VARIANT_QMV: return qmv_describe(a, buf, buflen);
        case AQ_VARIANT_TC: return tc_describe(a, buf, buflen);
        case AQ_VARIANT_TCW: return tcw_describe(a, buf, buflen);
        default: return snprintf(buf, buflen, "generic");
    }
}

int aq_attention_describe(int64_t H, int64_t KV, int64_t N, int64_t D, int bits, int group_size,
                          char *buf, int buflen) {
    if (!buf || buflen < 1) return -1;
    if (H < 1 || KV < 1 || N < 1 || H % KV != 0) return snprintf(buf, buflen, "invalid arguments");
    if (!attention_supported(H, KV, N, D, bits, group_size))
        return snprintf(buf, buflen, "unsupported");
    return attention_describe(H, KV, N, D, bits, group_size, 0, buf, buflen);
}

int aq_attention_describe_ws(int64_t H, int64_t KV, int64_t N, int64_t D, int bits,
                             int group_size, size_t workspace_bytes, char *buf, int buflen) {
    if (!buf || buflen < 1) return -1;
    if (H < 1 || KV < 1 || N < 1 || H % KV != 0) return snprintf(buf, buflen, "invalid arguments");
    if (!attention_supported(H, KV, N, D, bits, group_size))
        return snprintf(buf, buflen, "unsupported");
    return attention_describe(H, KV, N, D, bits, group_size, workspace_bytes, buf, buflen);
}

aq_status aq_stats(uint64_t *calls, int n) {
    if (n < 0 || (n > 0 && !calls)) return AQ_ERR_INVALID_ARG;
    for (int v = 0; v < AQ_NUM_VARIANTS && v < n; ++v) calls[v] = g_calls[v].load();
    return AQ_OK;
}

void aq_stats_reset(void) {
    for (auto &c : g_calls) c.store(0);
}

aq_status aq_device_error(uint32_t *code, int clear) {
    if (!code) return AQ_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return AQ_ERR_CUDA;
    uint32_t a = 0, b = 0, c = 0, d = 0;
    if (qmv_read_error(&a, clear != 0) != cudaSuccess) return AQ_ERR_CUDA;
    if (tc_read_error(&b, clear != 0) != cudaSuccess) return AQ_ERR_CUDA;
    if (gemv_read_error(&c, clear != 0) != cudaSuccess) return AQ_ERR_CUDA;
    if (attn_read_error(&d, clear != 0) != cudaSuccess) return AQ_ERR_CUDA;
    *code = a | b | c | d;
    return AQ_OK;
}

void aq_free(void) {
    for (auto &c : g_sms_cache) c.store(0);
}

const char *aq_status_string(aq_status status) {
    switch (status) {
        case AQ_OK: return "ok";
        case AQ_ERR_INVALID_ARG: return "invalid argument";
        case AQ_ERR_UNSUPPORTED: return "unsupported shape or variant";
        case AQ_ERR_MISALIGNED: return "misaligned pointer";
        case AQ_ERR_CUDA: return "CUDA runtime error";
        case AQ_ERR_NOMEM: return "out of memory";
        case AQ_ERR_DEVICE: return "device-side error";
    }
    return "unknown status";
}

const char *aq_variant_name(int variant) {
    switch (variant) {
        case AQ_VARIANT_GENERIC: return "generic";
        case AQ_VARIANT_QMV: return "qmv";
        case AQ_VARIANT_TC: return "tc";
        case AQ_VARIANT_GEMV: return "gemv";
        case AQ_VARIANT_TCW: return "tcw";
    }
    return "?";
}

const char *aq_version(void) { return "aq 0.1.0 (sm_103a)"; }

#ifdef AQ_TEST_HOOKS
// Test builds only: make a producer withhold the copies of its first stage
// (see g_test_withhold), so that a test can watch a bounded wait run out.
void aq_test_withhold(int what) { aq::g_test_withhold = what; }
// Test builds only: force the tensor-core kernel's clustered K split to
// `ctas` CTAs sharing `tiles` tiles where that plan is valid (ctas = -1:
// never split this way; 0: the planner's choice).
void aq_test_cluster_split(int ctas, int tiles) {
    aq::g_test_cluster_split = ctas < 0 ? -1 : (ctas << 8) | (tiles & 255);
}
// Test builds only: co-resident clusters of 1..8 CTAs of the tensor-core
// kernel, as the planner sees them (out[c] for c = 1..8).
void aq_test_active_clusters(int *out) {
    const int *n = aq::tc_active_clusters_for_tests();
    for (int c = 1; c <= 8; ++c) out[c] = n[c];
}
// Test builds only: the tensor-core kernel's plan for these sizes, whatever
// the dispatch rule would pick.
int aq_test_describe_tc(int64_t M, int64_t N, int64_t K, int bits, int dtype, char *buf,
                        int buflen) {
    if (!buf || buflen < 1) return -1;
    const uintptr_t fake = 0x100000;
    aq::MatmulArgs a = aq::make_args(dtype, (const void *)fake, (const uint32_t *)fake,
                                     (const void *)fake, (const void *)fake, M, N, K, bits,
                                     (void *)fake, nullptr);
    if (aq::check_args(a) != AQ_OK) return snprintf(buf, buflen, "invalid arguments");
    return aq::tc_describe(a, buf, buflen);
}
#endif

}  // extern "C"
