/*
 * aq.h — C ABI of libaq: y = x . W^T over MLX-style affine group-64 weights
 * at 3 or 4 bits, on one NVIDIA GB300 (sm_103a).  Around it: packing and the
 * float -> affine quantiser, several projections of one x per call (q/k/v,
 * gate/up with SiLU), other code widths and group sizes, and decode
 * attention over a KV cache stored in the same format.
 *
 * Weight format (mlx-bun pages, @mlx-bun/inference 1.0.0,
 * kernels/quantization/affine-split-mma.ts helper affine_unit and
 * affine3-mma.ts / affine4-mma.ts helpers affine_q3 / affine_q4):
 *   - W has N rows of K values; K is a multiple of 64 (one group = 64 values);
 *   - a row's codes form one LSB-first bit stream: code v occupies bits
 *     [v*bits, v*bits + bits); stream bit i is bit i%32 of uint32 word i/32;
 *     so one group is 2*bits words and a row is K*bits/32 words (row-major
 *     [N][K*bits/32]); 3-bit codes may straddle two words;
 *   - scales and biases are fp16 [N][K/64]; a weight dequantises to
 *     w[n][k] = scale[n][k/64] * q[n][k] + bias[n][k/64].
 *
 * Conventions shared by every entry point:
 *   - Pointers named *_dev are DEVICE pointers (cudaMalloc / torch tensors);
 *     pointers named *_host are HOST pointers.  The caller owns all memory;
 *     the library borrows pointers until the work queued on `stream`
 *     completes and never frees them.  Arrays are dense and row-major.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is queued asynchronously; no entry point synchronises
 *     the device except aq_matmul_host (which synchronises `stream`) and
 *     aq_device_error.
 *   - The library allocates no device memory in any entry point (the
 *     fixed scratch of aq_attention_decode_static exists from module load).
 *   - Arguments are validated before anything is queued; a bad argument
 *     returns an error status and queues nothing.  Launch failures return
 *     AQ_ERR_CUDA.  Faults that happen later on the device surface at the
 *     caller's next synchronisation, as with any CUDA call.  Nothing prints.
 *   - Entry points are thread-safe when different threads use different
 *     streams; results do not depend on the thread or stream.
 *   - Results are deterministic: the same inputs give bit-identical outputs,
 *     call after call (fixed-order reductions, no atomics on data).
 *   - Consecutive matmul calls on one stream overlap (programmatic dependent
 *     launch): a call may start reading its Wq, scales and biases while the
 *     previous call on the stream is still running, and reads x and writes
 *     out only after that call has finished.  So the output of a matmul or
 *     attention call must not alias Wq_dev, scales_dev or biases_dev of the
 *     next matmul call on the same stream; everything else follows stream
 *     order (aq_attention_decode reads nothing before the previous call has
 *     finished).
 */
#ifndef AQ_H
#define AQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum aq_status {
    AQ_OK = 0,
    AQ_ERR_INVALID_ARG = 1, /* null pointer, negative size, bits not 3/4, K % 64 != 0 */
    AQ_ERR_UNSUPPORTED = 2, /* valid but not served (e.g. an explicit variant that cannot run this shape) */
    AQ_ERR_MISALIGNED = 3,  /* a pointer is not aligned to its element size */
    AQ_ERR_CUDA = 4,        /* a CUDA runtime call failed (launch, copy, attribute) */
    AQ_ERR_NOMEM = 5,       /* reserved: the library allocates nothing today */
    AQ_ERR_DEVICE = 6       /* a kernel reported a device-side error (see aq_device_error) */
} aq_status;

/* Element type of x and y. */
typedef enum aq_dtype { AQ_F16 = 0, AQ_BF16 = 1 } aq_dtype;

/* Kernel variants, for aq_matmul_variant, aq_select and aq_stats. */
typedef enum aq_variant {
    AQ_VARIANT_AUTO = -1,   /* the dispatch rule picks */
    AQ_VARIANT_GENERIC = 0, /* plain-load CUDA-core kernel: any K % 64 == 0, any alignment */
    AQ_VARIANT_QMV = 1,     /* small-M: bulk-async staged weights, warp MMA, factored dequant */
    AQ_VARIANT_TC = 2,      /* M > 32: tcgen05 MMA with TMEM accumulators; with fewer
                               weight tiles than SMs, a tile's K range shared over the
                               CTAs of a cluster */
    AQ_VARIANT_GEMV = 3,    /* M <= 32: one resident CTA per SM, TMA weight ring, warp MMA */
    AQ_VARIANT_TCW = 4,     /* M <= 128 (explicit only: the dispatch rule prefers TC):
                               tcgen05 MMA with x as the 128-row operand and 256-row
                               weight tiles, K split over a cluster */
    AQ_NUM_VARIANTS = 5
} aq_variant;

/*
 * aq_pack — pack integer codes into the bit stream described above.
 *   codes_dev  uint8 [N][K], device; only the low `bits` bits of each code
 *              are used (higher bits are ignored).
 *   words_dev  uint32 [N][K*bits/32], device, written entirely.
 * bits may be 2, 3, 4, 5, 6 or 8 (the same LSB-first stream; the matmul
 * takes 3 and 4 at groups of 64 in aq_matmul and the others in
 * aq_matmul_ex).
 * Errors: AQ_ERR_INVALID_ARG if N < 0, K < 0, K % 32 != 0, bits outside that
 * set, or a pointer is NULL while N*K > 0; AQ_ERR_MISALIGNED if words_dev is
 * not 4-byte aligned.  N == 0 or K == 0 queues nothing and returns AQ_OK.
 */
aq_status aq_pack(const uint8_t *codes_dev, int64_t N, int64_t K, int bits,
                  uint32_t *words_dev, void *stream);

/*
 * aq_quantize — quantise float weights W[N][K] (fp16) into the format above:
 * packed codes, one fp16 scale and one fp16 bias per 64-value group.
 * aq_quantize_bf16 — the same with bf16 weights.
 *   w_dev       [N][K] weights, device, 16-byte aligned, row-major.
 *   Wq_dev      uint32 [N][K*bits/32], device, caller-allocated, written entirely.
 *   scales_dev  fp16 [N][K/64], device, caller-allocated, written entirely.
 *   biases_dev  fp16 [N][K/64], device, caller-allocated, written entirely.
 * The pages define the format and w = scale*q + bias (affine-split-mma.ts,
 * helper affine_unit) but no quantiser; the rule here, decided in single
 * precision per group, is: scale = fp16((max - min) / (2^bits - 1)),
 * bias = fp16(min), q = clamp(rint((w - bias) / scale), 0, 2^bits - 1)
 * (q = 0 when the scale is 0); fp16 rounding is to nearest even.  Weights
 * must be finite and within fp16 range (the stored scale and bias are fp16).
 * Errors: AQ_ERR_INVALID_ARG if N < 0, K < 0, K % 64 != 0, bits not in
 * {3,4} or a pointer is NULL while N*K > 0; AQ_ERR_MISALIGNED if w_dev is not
 * 16-byte aligned, Wq_dev not 4-byte or scales/biases not 2-byte aligned;
 * AQ_ERR_CUDA if the launch fails.  N == 0 or K == 0 queues nothing.
 */
aq_status aq_quantize(const void *w_dev, int64_t N, int64_t K, int bits, uint32_t *Wq_dev,
                      void *scales_dev, void *biases_dev, void *stream);
aq_status aq_quantize_bf16(const void *w_dev, int64_t N, int64_t K, int bits,
                           uint32_t *Wq_dev, void *scales_dev, void *biases_dev, void *stream);

/*
 * aq_matmul — y[M][N] = x[M][K] . dequant(W)^T with fp16 x and fp16 y.
 * aq_matmul_bf16 — the same with bf16 x and bf16 y.
 *   x_dev      [M][K] activations, device.
 *   Wq_dev     uint32 [N][K*bits/32] packed codes, device.
 *   scales_dev fp16 [N][K/64], device.   biases_dev fp16 [N][K/64], device.
 *   out_dev    [M][N], device, caller-allocated; every element is written,
 *              nothing outside it is.
 * Accumulation is in fp32 and y is rounded to nearest even.  Any M >= 1,
 * N >= 1 and K >= 64 with K % 64 == 0 is served; the fast kernels also want
 * K % 512 == 0 and 16-byte aligned x, Wq, scales, biases and y (other
 * shapes go to the generic kernel).
 * Errors: AQ_ERR_INVALID_ARG if M < 1, N < 1, K < 64, K % 64 != 0, bits not
 * in {3,4} or a pointer is NULL; AQ_ERR_MISALIGNED if a pointer is not
 * aligned to its element size (2 bytes for x/y/scales/biases, 4 for Wq);
 * AQ_ERR_CUDA if a launch fails.
 * Follows affineSplitMma (affine-split-mma.ts): x of any row count times
 * W^T, y in x's dtype, rows past M never written.
 */
aq_status aq_matmul(const void *x_dev, const uint32_t *Wq_dev, const void *scales_dev,
                    const void *biases_dev, int64_t M, int64_t N, int64_t K, int bits,
                    void *out_dev, void *stream);
aq_status aq_matmul_bf16(const void *x_dev, const uint32_t *Wq_dev, const void *scales_dev,
                         const void *biases_dev, int64_t M, int64_t N, int64_t K, int bits,
                         void *out_dev, void *stream);

/*
 * aq_matmul_ex — aq_matmul for other code widths and group sizes: bits in
 * {2, 3, 4, 5, 6, 8}, groups of group_size in {32, 64, 128} values (the
 * pages' fused-decode kernel takes 4 and 8 bits with groups of 32, 64 and
 * 128).  Wq_dev is the same LSB-first stream (aq_pack), scales and biases
 * fp16 [N][K/group_size]; dtype AQ_F16 or AQ_BF16 for x and y.  3 and 4 bits
 * at groups of 64 run exactly as aq_matmul / aq_matmul_bf16 (the fast
 * kernels).  Otherwise: for M > 4 with K % 512 == 0 and x, Wq, scales and
 * biases 16-byte aligned, the tensor-core kernel with a dequantisation for
 * any width (counted under AQ_VARIANT_TC); at M <= 32 with x 16-byte aligned
 * (and the staged rows of x within 200 KB of shared memory) the small-M
 * segment kernel; anything else the plain kernel (both counted under
 * AQ_VARIANT_GENERIC).  Tolerance, ownership and errors as aq_matmul, with
 * K % group_size == 0 in place of K % 64 == 0.
 */
aq_status aq_matmul_ex(int dtype, const void *x_dev, const uint32_t *Wq_dev,
                       const void *scales_dev, const void *biases_dev, int64_t M, int64_t N,
                       int64_t K, int bits, int group_size, void *out_dev, void *stream);

/*
 * aq_quantize_ex — aq_quantize / aq_quantize_bf16 (dtype AQ_F16 / AQ_BF16)
 * for other code widths and group sizes (as aq_matmul_ex), with the same
 * rule per group; codes decided with the IEEE quotient in single precision.
 * w_dev 2-byte aligned; scales/biases fp16 [N][K/group_size].  Errors as
 * aq_quantize with K % group_size == 0.
 */
aq_status aq_quantize_ex(int dtype, const void *w_dev, int64_t N, int64_t K, int bits,
                         int group_size, uint32_t *Wq_dev, void *scales_dev, void *biases_dev,
                         void *stream);

/*
 * aq_attention_decode — decode attention over a quantised KV cache, one
 * query row per head (grouped-query):
 *   o[h] = softmax(q[h] . Kd[kv]^T) . Vd[kv],   kv = h / (H / KV),
 * Kd, Vd the caches dequantised as scale * code + bias per group of
 * group_size values along the head dimension.  This is the operator of the
 * fused decode kernel of the mlx-bun 0.0.4 page
 * (src/model/fused-decode-kernel.ts); the query is used as given (a
 * 1/sqrt(D) factor, if wanted, is folded into q by the caller, as the
 * pages' kernel expects a pre-scaled query).
 *   dtype         AQ_F16 or AQ_BF16: the type of q and o.
 *   q_dev         [H][D], device.
 *   k_words_dev   uint32 [KV][N][D*bits/32], device, 16-byte aligned: row
 *                 (kv, n) packed as aq_pack packs a weight row.
 *   k_scales_dev, k_biases_dev  fp16 [KV][N][D/group_size], device,
 *                 16-byte aligned.
 *   v_words_dev, v_scales_dev, v_biases_dev  the same for V.
 *   out_dev       o [H][D], device, caller-allocated.
 * Served: bits 4 or 8, group_size 32/64/128 (D % group_size == 0), D in
 * {64, 128, 256, 512}, H/KV in {1, 2, 4, 8}, any N >= 1.  Scores are fp32; the
 * probabilities times the value scales enter the value product as fp16
 * (relative error 2^-11 per term); o is rounded once.  The rows of a KV
 * head are split over the CTAs of one thread-block cluster and merged in
 * rank order (deterministic); the library allocates nothing.
 * Errors: AQ_ERR_INVALID_ARG for bad sizes, widths, group sizes or NULL
 * pointers; AQ_ERR_MISALIGNED; AQ_ERR_UNSUPPORTED for valid arguments
 * outside the served set (nothing queued); AQ_ERR_CUDA if the launch fails.
 */
aq_status aq_attention_decode(int dtype, const void *q_dev, const uint32_t *k_words_dev,
                              const void *k_scales_dev, const void *k_biases_dev,
                              const uint32_t *v_words_dev, const void *v_scales_dev,
                              const void *v_biases_dev, int64_t H, int64_t KV, int64_t N,
                              int64_t D, int bits, int group_size, void *out_dev, void *stream);

/*
 * aq_attention_describe — one line naming the geometry aq_attention_decode
 * launches for these sizes: "attn cluster=C block=R stages=S smem=B grid=G"
 * (C CTAs per KV head, R cached rows per CTA, S stages in the shared-memory
 * ring, B bytes of dynamic shared memory).  Queries the current device for
 * co-resident clusters; "no device" without one, "unsupported" or "invalid
 * arguments" for sizes aq_attention_decode would refuse.  Writes at most
 * buflen bytes (NUL-terminated) to the host buffer and returns the length it
 * wanted (as snprintf), or -1 if buf is NULL or buflen < 1.
 */
int aq_attention_describe(int64_t H, int64_t KV, int64_t N, int64_t D, int bits, int group_size,
                          char *buf, int buflen);

/*
 * aq_attention_workspace_bytes — the workspace aq_attention_decode_ws needs
 * to spread each KV head's rows over several thread-block clusters (the
 * pages' kernel splits the rows of a head into blocks merged afterwards:
 * src/model/fused-decode-kernel.ts, the flash-decoding split and its
 * deterministic merge).  Returns 0 when one cluster per KV head is the best
 * plan for these sizes on the current device, or for arguments
 * aq_attention_decode would refuse.
 */
size_t aq_attention_workspace_bytes(int64_t H, int64_t KV, int64_t N, int64_t D, int bits,
                                    int group_size);

/*
 * aq_attention_decode_ws — aq_attention_decode with a caller-provided
 * workspace, so that a KV head's rows may span several clusters and the
 * kernel may hold every SM (one cluster per KV head can hold only as many
 * CTAs as the largest co-resident cluster).  Each cluster merges its CTAs in
 * rank order through distributed shared memory and writes its partial
 * (max, sum, unnormalised o per query head) to the workspace; the cluster
 * that arrives last at a per-KV-head counter (one atomic add per cluster, no
 * waiting) adds the partials in cluster order, writes o, and sets the
 * counter back to zero.  The result is deterministic (fixed merge order)
 * but not bit-identical to aq_attention_decode's (another split).
 *   workspace_dev    device, 256-byte aligned, workspace_bytes long,
 *                    owned by the caller.  Its first KV 32-bit words (the
 *                    counters) must be zero before the first call (e.g.
 *                    allocate it zeroed); every call leaves them zero.  The
 *                    rest needs no initial value.
 *   workspace_bytes  at least aq_attention_workspace_bytes(...) to get the
 *                    several-cluster plan; any smaller size (0 with a NULL
 *                    workspace) runs the one-cluster plan, as
 *                    aq_attention_decode.
 * Calls that may overlap (other streams, or the same workspace in flight)
 * must use distinct workspaces.  Other arguments, results and errors as
 * aq_attention_decode; AQ_ERR_INVALID_ARG also for workspace_bytes > 0 with
 * a NULL workspace, AQ_ERR_MISALIGNED for a workspace not 256-byte aligned.
 */
aq_status aq_attention_decode_ws(int dtype, const void *q_dev, const uint32_t *k_words_dev,
                                 const void *k_scales_dev, const void *k_biases_dev,
                                 const uint32_t *v_words_dev, const void *v_scales_dev,
                                 const void *v_biases_dev, int64_t H, int64_t KV, int64_t N,
                                 int64_t D, int bits, int group_size, void *out_dev,
                                 void *workspace_dev, size_t workspace_bytes, void *stream);

/*
 * aq_attention_decode_static — aq_attention_decode_ws without a caller
 * workspace: the several-cluster plan's workspace is a fixed array of
 * AQ_ATTENTION_STATIC_SCRATCH_BYTES in device memory the library owns, so
 * the call allocates nothing, for hosts that cannot allocate device memory
 * per call (a C caller with no device allocator of its own, a decode loop
 * that must not synchronise on cudaMalloc).  The pages have no counterpart
 * (their kernel sums the blocks through a framework array); this is an
 * interface of this library only.
 *   Arguments, results and errors as aq_attention_decode, and the same plan
 *   and results as aq_attention_decode_ws given a workspace of
 *   aq_attention_workspace_bytes(...): AQ_ERR_UNSUPPORTED (nothing queued)
 *   also when that workspace is larger than the array.
 *   The array is zero at module load and every call leaves its counters
 *   zero.  Its device address is looked up once per device on the first
 *   call that needs it (cudaGetSymbolAddress): make that first call outside
 *   stream capture.  One array per device: calls that may overlap in time
 *   on one device (other streams, other host threads) share it and race; the
 *   caller serialises them.
 */
#define AQ_ATTENTION_STATIC_SCRATCH_BYTES 1048576
aq_status aq_attention_decode_static(int dtype, const void *q_dev, const uint32_t *k_words_dev,
                                     const void *k_scales_dev, const void *k_biases_dev,
                                     const uint32_t *v_words_dev, const void *v_scales_dev,
                                     const void *v_biases_dev, int64_t H, int64_t KV, int64_t N,
                                     int64_t D, int bits, int group_size, void *out_dev,
                                     void *stream);

/*
 * aq_attention_describe_ws — aq_attention_describe for
 * aq_attention_decode_ws with a workspace of workspace_bytes: with a
 * workspace the line also names "clusters_per_kv_head=K workspace=W" (the
 * grid is KV x C x K CTAs, W the bytes the plan uses).
 */
int aq_attention_describe_ws(int64_t H, int64_t KV, int64_t N, int64_t D, int bits,
                             int group_size, size_t workspace_bytes, char *buf, int buflen);

/* Largest number of projections aq_matmul_multi takes in one call. */
#define AQ_MAX_PROJ 4

/*
 * aq_matmul_multi — several projections of the same activations in one call:
 * y_j[M][N[j]] = x[M][K] . dequant(W_j)^T for j < nproj (1..AQ_MAX_PROJ),
 * all with the same K and bits, e.g. the q, k and v projections of a
 * decoder layer.  The small projections then share one launch instead of
 * each paying its own (the pages' fused multi-projection decode idea).
 *   dtype       AQ_F16 or AQ_BF16: the type of x and of every y_j.
 *   Wq_dev, scales_dev, biases_dev, out_dev, N: host arrays of nproj
 *               entries; entry j is projection j, laid out and owned as in
 *               aq_matmul (device pointers, out caller-allocated).
 * M <= 32 with K % 512 == 0 and 16-byte alignment runs as one launch of the
 * resident small-M kernel; anything else runs one launch per projection
 * under the usual dispatch rule, with the same results.  Outputs must not
 * overlap each other, x or the weights.
 * Errors: AQ_ERR_INVALID_ARG for a bad dtype, nproj outside 1..AQ_MAX_PROJ,
 * a NULL array, or any projection that aq_matmul would reject; otherwise as
 * aq_matmul.
 */
aq_status aq_matmul_multi(int dtype, const void *x_dev, int nproj,
                          const uint32_t *const *Wq_dev, const void *const *scales_dev,
                          const void *const *biases_dev, const int64_t *N, int64_t M,
                          int64_t K, int bits, void *const *out_dev, void *stream);

/*
 * aq_matmul_gate_up — the gated MLP input of a decoder layer in one call:
 * h[M][N] = silu(x . dequant(W_gate)^T) * (x . dequant(W_up)^T), with
 * silu(g) = g / (1 + exp(-g)), both products accumulated in fp32 and h
 * rounded once to x's dtype (the pages' fused gate/up + SiLU epilogue).
 * Every CTA decodes the same rows of both projections, so the gate value
 * never leaves the SM.  Both weight sets are [N][K] as in aq_matmul.
 *   dtype    AQ_F16 or AQ_BF16 (x and h).
 *   out_dev  h [M][N], device, caller-allocated.
 * Served for M <= 32, K % 512 == 0, 16-byte alignment and N up to 128 rows
 * per SM (19456 on 152 SMs); otherwise AQ_ERR_UNSUPPORTED and nothing is
 * queued.  Errors otherwise as aq_matmul.
 */
aq_status aq_matmul_gate_up(int dtype, const void *x_dev, const uint32_t *Wg_dev,
                            const void *scales_g_dev, const void *biases_g_dev,
                            const uint32_t *Wu_dev, const void *scales_u_dev,
                            const void *biases_u_dev, int64_t M, int64_t N, int64_t K,
                            int bits, void *out_dev, void *stream);

/*
 * aq_matmul_variant — aq_matmul / aq_matmul_bf16 with the element type as an
 * argument and, optionally, an explicit kernel variant (AQ_VARIANT_AUTO lets
 * the dispatch rule choose).  An explicit variant that cannot run the shape
 * or alignment returns AQ_ERR_UNSUPPORTED and queues nothing.  Same
 * arguments, ownership and errors as aq_matmul otherwise.
 */
aq_status aq_matmul_variant(int variant, int dtype, const void *x_dev, const uint32_t *Wq_dev,
                            const void *scales_dev, const void *biases_dev, int64_t M,
                            int64_t N, int64_t K, int bits, void *out_dev, void *stream);

/*
 * aq_matmul_host — the whole call from host memory: copies x_host to the
 * caller's device buffer x_dev, runs the matmul (auto dispatch) into out_dev,
 * copies the result back to out_host, and synchronises `stream`.
 *   x_host   [M][K] of `dtype`, host (pinned memory makes the copies async).
 *   x_dev    [M][K] device scratch owned by the caller.
 *   out_dev  [M][N] device scratch owned by the caller.
 *   out_host [M][N] of `dtype`, host, written on return.
 * Weights (Wq_dev, scales_dev, biases_dev) stay resident on the device.
 * Errors: as aq_matmul, plus AQ_ERR_CUDA if a copy or the synchronisation
 * fails.
 */
aq_status aq_matmul_host(int dtype, const void *x_host, const uint32_t *Wq_dev,
                         const void *scales_dev, const void *biases_dev, int64_t M, int64_t N,
                         int64_t K, int bits, void *out_host, void *x_dev, void *out_dev,
                         void *stream);

/*
 * aq_select — the variant the dispatch rule picks for a shape, without
 * launching anything (host logic only; needs no GPU).  Alignment is assumed
 * to be 16 bytes.  Returns an aq_variant value, or -1 for invalid arguments.
 */
int aq_select(int64_t M, int64_t N, int64_t K, int bits, int dtype);

/*
 * aq_describe — one line of text naming the kernel and launch geometry the
 * dispatch rule picks for a shape (host logic only; needs no GPU).  Writes a
 * NUL-terminated string of at most buflen bytes to the host buffer `buf` and
 * returns the length it wanted (as snprintf), or -1 if buf is NULL or
 * buflen < 1.
 */
int aq_describe(int64_t M, int64_t N, int64_t K, int bits, int dtype, char *buf, int buflen);

/*
 * aq_stats — per-variant call counters since load (or the last
 * aq_stats_reset), so a caller or a test can assert which kernel actually
 * ran.  This follows the dispatch counter of the mlx-bun 0.0.4 page
 * (src/model/fused-decode-kernel.ts, fusedKernelCalls, which a gate test
 * reads to confirm the fused kernel ran), kept per variant here.
 *   calls  host array of n uint64; element v receives the number of calls
 *          that launched variant v (n may be less than AQ_NUM_VARIANTS;
 *          variants past n are not reported).
 * Errors: AQ_ERR_INVALID_ARG if n < 0, or calls is NULL while n > 0.
 * Counting is on the host at launch time (atomic, thread-safe).
 */
aq_status aq_stats(uint64_t *calls, int n);

/* aq_stats_reset — set every counter of aq_stats to zero. */
void aq_stats_reset(void);

/*
 * aq_device_error — read the device-side error word that kernels set when a
 * bounded wait gives up (a pipeline barrier not completing within its time
 * limit).  Synchronises the device first.  *code receives 0 when no error
 * was recorded; non-zero values identify the wait that gave up.  clear != 0
 * resets the word to 0.
 */
aq_status aq_device_error(uint32_t *code, int clear);

/*
 * aq_free — release library-held resources (cached device attributes and
 * kernel configuration state).  The pages' host wrapper (affineSplitMma in
 * affine-split-mma.ts) borrows its inputs and returns an array the caller
 * owns, so nothing the caller passes is ever freed by the library; this
 * call releases only what the library keeps for itself.  It holds no device
 * allocations; calling aq_free is optional and the library stays usable
 * afterwards (state is rebuilt on the next call).
 */
void aq_free(void);

/*
 * aq_status_string — human-readable name of a status code (static storage,
 * never NULL; "unknown status" for values outside aq_status).  The pages'
 * host wrapper reports a bad call by throwing with a message (affineSplitMma
 * throws "no rows" for M < 1); a C ABI returns the status instead and this
 * gives its text.
 */
const char *aq_status_string(aq_status status);

/* Human-readable name of a variant ("generic", "qmv", "tc", "gemv", "tcw"); "?" if unknown. */
const char *aq_variant_name(int variant);

/* Library version string. */
const char *aq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* AQ_H */
