// Resident small-M kernel: plan, tensor maps and launch.  The kernel itself
// (and its design notes) is in aq_gemv.cuh; the two-column-block
// instantiations are in aq_gemv16.cu.
#include "aq_gemv.cuh"

namespace aq {

__device__ uint32_t g_gemv_error;

namespace gemv {
namespace {

uint32_t round_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

// Largest whole-x footprint (rows of x, group sums and scales) kept in
// shared memory; beyond it x is streamed with the weights.  A 13824-long
// row (27.6 KB + 13.8 KB of sums and scales) still fits.
constexpr size_t kXWholeMax = 48 * 1024;

// Shared-memory budget of a plan (AQ_GEMV_SMEM_KB overrides it for
// experiments).
size_t smem_budget() {
    static const size_t v = [] {
        const char *e = std::getenv("AQ_GEMV_SMEM_KB");
        const long kb = (e && *e) ? std::atol(e) : 0;
        return kb > 0 ? std::min<size_t>((size_t)kb * 1024, kSmemMax) : kSmemBudget;
    }();
    return v;
}

// Groups per warp per stage (the units of a stage are unrolled; this bounds
// code and registers), by tiles per pass and column blocks.
int max_wps(int tiles, int mb) {
    if (mb > 2) return 1;
    if (mb > 1) return tiles <= 2 ? 2 : 1;
    return tiles <= 2 ? 4 : tiles <= 4 ? 2 : 1;
}

uint32_t *error_word() {
    static uint32_t *ptr = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_gemv_error) == cudaSuccess)
            ptr = static_cast<uint32_t *>(p);
        else
            cudaGetLastError();
    });
    return ptr;
}

// The plan of a launch.  Several projections of the same x (n_proj[0..nproj),
// a.N unused): their rows are split evenly over the SMs, each CTA within one
// projection.  gate_up: two projections of a.N rows, every CTA the same rows
// of both (two passes).
bool gemv_plan(const MatmulArgs &a, GemvPlan &pl, const int64_t *n_proj, int nproj,
               bool gate_up) {
    if (nproj < 1 || nproj > kMaxProj || (gate_up && nproj != 2)) return false;
    int64_t n_rows = a.N;
    if (nproj > 1 && !gate_up) {
        n_rows = 0;
        for (int j = 0; j < nproj; ++j) {
            if (n_proj[j] < 1 || n_proj[j] > INT32_MAX / 2) return false;
            n_rows += n_proj[j];
        }
    }
    if (a.M < 1 || a.M > 32 || n_rows < 1 || a.K < 512 || a.K % 512 != 0) return false;
    if (n_rows > INT32_MAX / 2) return false;
    if (a.K > INT32_MAX / 2) return false;
    const int B = a.bits;
    const int G = (int)(a.K / 64);
    const int MB = a.M > 16 ? 4 : a.M > 8 ? 2 : 1;
    const int max_tiles = MB == 1 ? kMaxTiles : 6;
    // Two or four column blocks take too many registers for two CTAs per SM:
    // the CTA has the SM to itself and all of its shared memory.
    const size_t budget = MB > 1 ? kSmemMax : smem_budget();
    const int sms = num_sms();
    const int64_t per_sm = (n_rows + sms - 1) / sms;
    int passes = (int)((per_sm + 16 * max_tiles - 1) / (16 * max_tiles));
    int pr = (int)((per_sm + passes - 1) / passes);
    int64_t rows_cta = (int64_t)pr * passes;
    if (gate_up) {  // pass 0 the gate, pass 1 the up rows, the same rows
        if (per_sm > 16 * max_tiles) return false;
        passes = 2;
        pr = (int)per_sm;
        rows_cta = pr;
    }
    GemvParams &q = pl.prm;
    q.M = (int)a.M;
    q.N = (int)n_rows;
    q.K = (int)a.K;
    q.rows_cta = (int)rows_cta;
    q.pass_rows = pr;
    q.passes = passes;
    q.tiles = (pr + 15) / 16;
    GemvMulti &mx = pl.mx;
    memset(&mx, 0, sizeof(mx));
    pl.mp = nproj > 1 || gate_up;
    mx.nproj = nproj;
    mx.gate_up = gate_up ? 1 : 0;
    if (nproj > 1 && !gate_up) {
        int c = 0;
        for (int j = 0; j < nproj; ++j) {
            mx.cta0[j] = c;
            mx.n_proj[j] = (int)n_proj[j];
            c += (int)((n_proj[j] + rows_cta - 1) / rows_cta);
        }
        mx.cta0[nproj] = c;
        pl.grid = c;
    } else {
        pl.grid = (int)((a.N + rows_cta - 1) / rows_cta);
        mx.cta0[0] = 0;
        mx.cta0[1] = pl.grid;
        mx.n_proj[0] = mx.n_proj[1] = (int)a.N;
    }
    const uint32_t rows_pad = 16u * (uint32_t)q.tiles;
    const uint32_t box = B == 4 ? 128u : 96u;
    pl.mb = MB;
    pl.bits = B;
    pl.bf16 = a.dtype == AQ_BF16;
    const uint32_t red_bytes = (uint32_t)kConsumers * q.tiles * MB * 32 * 4 * 4;
    const uint32_t gu_bytes = gate_up ? round_up((uint32_t)pr * (uint32_t)a.M * 4u, 128u) : 0u;

    // The widest stage (most groups per warp) that keeps at least three
    // stages in the ring (or the whole of K), else two; x whole in shared
    // memory (single column block only) before x staged with the weights.
    for (int want = 3; want >= 2; --want) {
        for (int whole = MB > 1 ? 0 : 1; whole >= 0; --whole) {
            for (int wps = max_wps(q.tiles, MB); wps >= 1; wps /= 2) {
                const int sg = 8 * wps;
                // a last stage past the end of K reads zeros and its groups are skipped
                q.sg = sg;
                q.n_stages = (G + sg - 1) / sg;
                const uint32_t nb = (uint32_t)sg / 4;
                // codes [nb][pr][box] and scales, biases [sg/8][pr][8], each with
                // room for the padded rows of the last block
                const uint32_t wbytes = round_up((nb * (uint32_t)pr + rows_pad - (uint32_t)pr) * box,
                                                 B == 4 ? 1024u : 128u);
                const uint32_t sbytes =
                    round_up(((nb / 2 - 1) * (uint32_t)pr + rows_pad) * 16u, 128u);
                q.off_sc = wbytes;
                q.off_bi = wbytes + sbytes;
                const int total = passes * q.n_stages;
                {
                    q.x_whole = whole;
                    q.x_row_pitch = (uint32_t)a.K * 2u + 16u;
                    // staged x: the stage's groups x M rows x 128 B, 1024-aligned
                    q.x_rows = (int)a.M;
                    const uint32_t xst = whole ? 0u : (uint32_t)sg * (uint32_t)a.M * 128u;
                    q.off_xst = round_up(q.off_bi + sbytes, 1024u);
                    q.slot_bytes = round_up(q.off_xst + xst, 1024u);
                    q.stage_tx =
                        nb * (uint32_t)pr * box + 2u * (uint32_t)pr * (uint32_t)sg * 2u + xst;
                    // whole x: rows at 2K + 16 bytes, then group sums and scales [2][G][8]
                    const size_t x_bytes =
                        whole ? round_up(q.x_row_pitch * (uint32_t)a.M, 128u) + (size_t)G * 64 : 0;
                    if (whole && x_bytes > kXWholeMax) continue;
                    const size_t bars = 2 * 8 * (size_t)total + 16 + 16;
                    // With one pass the partial tiles reuse the ring if it is large enough.
                    for (int alias = passes == 1 ? 1 : 0; alias >= 0; --alias) {
                        const size_t fixed = x_bytes + (alias ? 0 : red_bytes) + gu_bytes + bars +
                                             1024 /* alignment */;
                        if (fixed >= budget) continue;
                        const int ring =
                            (int)std::min<size_t>((size_t)total, (budget - fixed) / q.slot_bytes);
                        if (ring < std::min(want, total)) continue;
                        if (alias && (size_t)ring * q.slot_bytes < red_bytes) continue;
                        q.ring = ring;
                        q.red_alias = alias;
                        size_t off = (size_t)ring * q.slot_bytes;
                        q.off_x = (uint32_t)off;
                        q.off_xs = (uint32_t)(off + round_up(q.x_row_pitch * (uint32_t)a.M, 128u));
                        off += x_bytes;
                        q.off_red = alias ? 0u : (uint32_t)off;
                        off += alias ? 0 : red_bytes;
                        mx.off_gu = (uint32_t)off;
                        off += gu_bytes;
                        q.off_bar = (uint32_t)off;
                        off += 2 * 8 * (size_t)ring + 16 + 16;
                        pl.smem = off + 1024;
                        q.x = a.x;
                        q.y = a.out;
                        mx.y_proj[0] = a.out;
                        q.err = nullptr;
                        pl.wps = wps;
                        if (pl.smem <= budget) return true;
                    }
                }
            }
        }
    }
    return false;
}

}  // namespace
}  // namespace gemv

using gemv::GemvPlan;
using gemv::gemv_plan;

bool gemv_supported(const MatmulArgs &a) {
    if (!aligned(a.x, 16) || !aligned(a.Wq, 16) || !aligned(a.scales, 16) ||
        !aligned(a.biases, 16))
        return false;
    GemvPlan pl;
    return gemv_plan(a, pl, nullptr, 1, false);
}

namespace {

// Tensor maps for the plan and launch.  Projection j's codes, scales and
// biases are Wq[j], sc[j], bi[j] with n[j] rows.
cudaError_t launch_plan(const MatmulArgs &a, GemvPlan &pl, const uint32_t *const *Wq,
                        const void *const *sc, const void *const *bi, const int64_t *n,
                        int nproj) {
    const uint64_t row_bytes = (uint64_t)a.K * a.bits / 8, G = (uint64_t)a.K / 64;
    const uint32_t pr = (uint32_t)pl.prm.pass_rows, sg = (uint32_t)pl.prm.sg;
    const uint64_t box = a.bits == 4 ? 128 : 96;
    gemv::GemvMaps maps;
    memset(&maps, 0, sizeof(maps));
    const bool staged = !pl.prm.x_whole;
    if (staged) {
        // x as [G][M][64] elements: one box = the stage's groups x M rows
        const uint64_t xdims[3] = {64, (uint64_t)a.M, G};
        const uint64_t xstrides[2] = {(uint64_t)a.K * 2, 128};
        const uint32_t xbox[3] = {64, (uint32_t)a.M, sg};
        if (!tmap_encode(&maps.x, a.dtype == AQ_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                         3, a.x, xdims, xstrides, xbox, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    for (int j = 0; j < nproj; ++j) {
        // codes as [row_bytes / box][N][box] bytes: one box = sg/4 column blocks x pr rows
        const uint64_t wdims[3] = {box, (uint64_t)n[j], row_bytes / box};
        const uint64_t wstrides[2] = {row_bytes, box};
        const uint32_t wbox[3] = {(uint32_t)box, pr, sg / 4};
        // scales, biases as [G / 8][N][8] halves: one box = sg/8 blocks of 8 groups x pr rows
        const uint64_t sdims[3] = {8, (uint64_t)n[j], G / 8};
        const uint64_t sstrides[2] = {2 * G, 16};
        const uint32_t sbox[3] = {8, pr, sg / 8};
        if (!tmap_encode(&maps.w[j], CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, Wq[j], wdims, wstrides,
                         wbox,
                         a.bits == 4 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !tmap_encode(&maps.s[j], CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, sc[j], sdims, sstrides,
                         sbox, CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !tmap_encode(&maps.b[j], CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, bi[j], sdims, sstrides,
                         sbox, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    }
    if (!staged) maps.x = maps.w[0];  // unused; any valid map
    for (int j = nproj; j < gemv::kMaxProj; ++j) {  // unused projections
        maps.w[j] = maps.w[0];
        maps.s[j] = maps.s[0];
        maps.b[j] = maps.b[0];
    }
    pl.prm.err = gemv::error_word();
#ifdef AQ_TEST_HOOKS
    pl.prm.withhold = g_test_withhold == 1;
#endif
    if (!pl.prm.err) return cudaErrorInvalidValue;
    using gemv::launch_blocks;
    if (pl.mp) {
        if (pl.mb > 2) return launch_blocks<4, true, true>(pl, maps, a.stream);
        if (pl.mb > 1) return launch_blocks<2, true, true>(pl, maps, a.stream);
        return staged ? launch_blocks<1, true, true>(pl, maps, a.stream)
                      : launch_blocks<1, false, true>(pl, maps, a.stream);
    }
    if (pl.mb > 2) return launch_blocks<4, true, false>(pl, maps, a.stream);
    if (pl.mb > 1) return launch_blocks<2, true, false>(pl, maps, a.stream);
    return staged ? launch_blocks<1, true, false>(pl, maps, a.stream)
                  : launch_blocks<1, false, false>(pl, maps, a.stream);
}

}  // namespace

cudaError_t gemv_launch(const MatmulArgs &a) {
    GemvPlan pl;
    if (!gemv_plan(a, pl, nullptr, 1, false)) return cudaErrorInvalidValue;
    const int64_t n = a.N;
    return launch_plan(a, pl, &a.Wq, &a.scales, &a.biases, &n, 1);
}

bool gemv_multi_supported(const MultiArgs &m) {
    if (!aligned(m.a.x, 16)) return false;
    for (int j = 0; j < m.nproj; ++j)
        if (!aligned(m.Wq[j], 16) || !aligned(m.scales[j], 16) || !aligned(m.biases[j], 16))
            return false;
    GemvPlan pl;
    return gemv_plan(m.a, pl, m.N, m.nproj, m.gate_up);
}

cudaError_t gemv_launch_multi(const MultiArgs &m) {
    GemvPlan pl;
    if (!gemv_plan(m.a, pl, m.N, m.nproj, m.gate_up)) return cudaErrorInvalidValue;
    for (int j = 0; j < m.nproj; ++j) pl.mx.y_proj[j] = m.gate_up ? m.a.out : m.out[j];
    pl.prm.y = pl.mx.y_proj[0];  // one projection: the single-projection kernels
    return launch_plan(m.a, pl, m.Wq, m.scales, m.biases, m.N, m.nproj);
}

int gemv_describe_multi(const MultiArgs &m, char *buf, int len) {
    GemvPlan pl;
    if (!gemv_plan(m.a, pl, m.N, m.nproj, m.gate_up)) return snprintf(buf, len, "gemv: unsupported");
    const gemv::GemvParams &q = pl.prm;
    return snprintf(buf, len,
                    "gemv %s projections=%d rows/cta=%d passes=%d tiles=%d colblocks=%d "
                    "groups/stage=%d stages=%d ring=%d x=%s grid=%d smem=%zu",
                    m.gate_up ? "gate_up" : "multi", m.nproj, q.rows_cta, q.passes, q.tiles, pl.mb,
                    q.sg, q.n_stages, q.ring, q.x_whole ? "whole" : "staged", pl.grid, pl.smem);
}

int gemv_describe(const MatmulArgs &a, char *buf, int len) {
    GemvPlan pl;
    if (!gemv_plan(a, pl, nullptr, 1, false)) return snprintf(buf, len, "gemv: unsupported");
    const gemv::GemvParams &q = pl.prm;
    return snprintf(buf, len,
                    "gemv rows/cta=%d passes=%d tiles=%d colblocks=%d groups/stage=%d stages=%d "
                    "ring=%d x=%s grid=%d smem=%zu",
                    q.rows_cta, q.passes, q.tiles, pl.mb, q.sg, q.n_stages, q.ring,
                    q.x_whole ? "whole" : "staged",
                    pl.grid, pl.smem);
}

cudaError_t gemv_read_error(uint32_t *code, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(code, g_gemv_error, sizeof(uint32_t));
    if (e != cudaSuccess || !clear) return e;
    const uint32_t zero = 0;
    return cudaMemcpyToSymbol(g_gemv_error, &zero, sizeof(uint32_t));
}

}  // namespace aq

namespace aq {
namespace gemv {
template cudaError_t launch_blocks<1, false, false>(const GemvPlan &, const GemvMaps &, cudaStream_t);
}  // namespace gemv
}  // namespace aq
