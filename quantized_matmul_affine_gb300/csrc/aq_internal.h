// Host-side declarations shared by the translation units of libaq.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/aq.h"

namespace aq {

struct MatmulArgs {
    const void *x;
    const uint32_t *Wq;
    const void *scales;
    const void *biases;
    void *out;
    int64_t M, N, K;
    int bits;
    int dtype;  // AQ_F16 / AQ_BF16
    cudaStream_t stream;
};

// Several projections of one x in one launch (aq_matmul_multi) or the fused
// gate/up pair (aq_matmul_gate_up: projection 0 the gate, 1 the up rows,
// a.N rows each, y = silu(gate) * up in a.out).  a.Wq / a.scales / a.biases
// are unused.
struct MultiArgs {
    MatmulArgs a;
    int nproj;
    bool gate_up;
    const uint32_t *Wq[4];
    const void *scales[4];
    const void *biases[4];
    void *out[4];
    int64_t N[4];
};

// Device-side error codes (the word read by aq_device_error).  The low byte
// names the kernel, the next byte the wait that gave up.
enum : uint32_t {
    ERR_QMV_FULL = 0x0101,
    ERR_QMV_EMPTY = 0x0201,
    ERR_TC_BASE = 0x0002,
    ERR_GEMV_FULL = 0x0103,
    ERR_GEMV_EMPTY = 0x0203,
    ERR_GEMV_DRAIN = 0x0303,
    ERR_ATTN_FULL = 0x0104,
    ERR_ATTN_EMPTY = 0x0204,
    ERR_ATTN_PAIR = 0x0304,
};

// Each returns cudaSuccess, or the launch error.  `supported` reports
// whether the variant can run the shape/alignment at all.
bool generic_supported(const MatmulArgs &a);
cudaError_t generic_launch(const MatmulArgs &a);

bool gemv_supported(const MatmulArgs &a);
cudaError_t gemv_launch(const MatmulArgs &a);
bool gemv_multi_supported(const MultiArgs &m);
cudaError_t gemv_launch_multi(const MultiArgs &m);
int gemv_describe_multi(const MultiArgs &m, char *buf, int len);
int gemv_describe(const MatmulArgs &a, char *buf, int len);

bool qmv_supported(const MatmulArgs &a);
cudaError_t qmv_launch(const MatmulArgs &a);
// Tuning hook: restrict the small-M kernel's geometry (0 = free choice).
void qmv_force_geometry(int rows_tiles, int cluster_split, int ring_depth);
int qmv_describe(const MatmulArgs &a, char *buf, int len);

bool tc_supported(const MatmulArgs &a);
bool tcw_supported(const MatmulArgs &a);
cudaError_t tcw_launch(const MatmulArgs &a);
int tcw_describe(const MatmulArgs &a, char *buf, int len);
cudaError_t tc_launch(const MatmulArgs &a);
// The tensor-core kernel for other code widths (2..8 bits) and group sizes
// (32/64/128): K % 512 == 0, x, Wq, scales and biases 16-byte aligned.
bool tc_supported_g(const MatmulArgs &a, int group);
cudaError_t tc_launch_g(const MatmulArgs &a, int group);
int tc_describe(const MatmulArgs &a, char *buf, int len);

cudaError_t quantize_launch(int dtype, const void *w, int64_t N, int64_t K, int bits,
                            uint32_t *words, void *scales, void *biases, cudaStream_t stream);
cudaError_t quantize_launch_g(int dtype, const void *w, int64_t N, int64_t K, int bits, int group,
                              uint32_t *words, void *scales, void *biases, cudaStream_t stream);
bool generic_supported_g(const MatmulArgs &a, int group);
// The small-M kernel of the other widths and group sizes (aq_segv.cu).
bool segv_supported(const MatmulArgs &a, int group);
cudaError_t segv_launch(const MatmulArgs &a, int group);
bool attention_supported(int64_t H, int64_t KV, int64_t N, int64_t D, int bits, int group);
// The launch geometry aq_attention_decode (ws_bytes 0) or
// aq_attention_decode_ws (a workspace of ws_bytes) would use (snprintf
// semantics).
int attention_describe(int64_t H, int64_t KV, int64_t N, int64_t D, int bits, int group,
                       size_t ws_bytes, char *buf, int len);
// Workspace bytes that let the attention kernel spread a KV head over
// several clusters (0 when one cluster a KV head is the best plan).
size_t attention_workspace_bytes(int64_t H, int64_t KV, int64_t N, int64_t D, int bits,
                                 int group);
// The library's static attention scratch on the current device (its
// address looked up once per device), or nullptr.
void *attention_static_scratch();
// ws: a workspace of ws_bytes (256-byte aligned; its counters zero), or null.
cudaError_t attention_launch(int dtype, const void *q, const uint32_t *kw, const void *ks,
                             const void *kb, const uint32_t *vw, const void *vs, const void *vb,
                             int64_t H, int64_t KV, int64_t N, int64_t D, int bits, int group,
                             void *out, void *ws, size_t ws_bytes, cudaStream_t stream);
cudaError_t generic_launch_g(const MatmulArgs &a, int group);
cudaError_t pack_launch(const uint8_t *codes, int64_t N, int64_t K, int bits, uint32_t *words,
                        cudaStream_t stream);

#ifdef AQ_TEST_HOOKS
// Test builds only (never in libaq.so): which producer withholds the copies
// of its first stage, so that the waits on them run out (1 = the resident
// small-M kernel, 2 = the large-M tensor-core kernel, 0 = none).
extern int g_test_withhold;
// Test builds only: the tensor-core kernel's clustered K split, forced to
// (CTAs << 8) | tiles a cluster where that plan is valid (-1: never; 0: the
// planner's choice).
extern int g_test_cluster_split;
const int *tc_active_clusters_for_tests();
#endif

// Device error words, one per translation unit that owns bounded waits.
cudaError_t gemv_read_error(uint32_t *code, bool clear);
cudaError_t qmv_read_error(uint32_t *code, bool clear);
cudaError_t tc_read_error(uint32_t *code, bool clear);
cudaError_t attn_read_error(uint32_t *code, bool clear);

// A tiled TMA tensor map of `rank` dimensions (dims[0] innermost, strides
// in bytes of dims 1..rank-1), box `box`, out-of-range elements read as
// zero.  False if the driver entry point is missing or rejects the layout.
bool tmap_encode(CUtensorMap *tm, CUtensorMapDataType type, int rank, const void *base,
                 const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box,
                 CUtensorMapSwizzle swizzle);
// The 2-D case: a row-major [dim1][dim0] array.
inline bool tmap_2d(CUtensorMap *tm, CUtensorMapDataType type, const void *base, uint64_t dim0,
                    uint64_t dim1, uint64_t row_stride_bytes, uint32_t box0, uint32_t box1,
                    CUtensorMapSwizzle swizzle) {
    const uint64_t dims[2] = {dim0, dim1};
    const uint64_t strides[1] = {row_stride_bytes};
    const uint32_t box[2] = {box0, box1};
    return tmap_encode(tm, type, 2, base, dims, strides, box, swizzle);
}

// Number of streaming multiprocessors of the current device (cached).
int num_sms();

inline bool aligned(const void *p, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

}  // namespace aq
