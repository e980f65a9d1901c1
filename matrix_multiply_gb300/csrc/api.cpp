// The C ABI of tcgemm: validation, normalisation, dispatch and launch.
//
// Call path of every GEMM (tessl architecture.md, "GEMM Pipeline & Kernel
// Selection" and "The Kernel Library and the nn Boundary"):
//   validate (checked sizes, dims, dtypes, leading dims, finite scalars,
//   overlap) -> normalise ld = 0 to contiguous (tensorcore gemm.md,
//   "Surface") -> plan (variant, tile, split, grid) -> repack operands TMA
//   cannot read -> encode TMA descriptors -> launch -> record the variant
//   (tensorcore gemm.md, "Fallback ladder": tc_last_backend).
// Nothing is enqueued unless every check passed.
#include "../../include/tcgemm.h"
#include "internal.h"

#include <cudaTypedefs.h>

#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <algorithm>
#include <atomic>
#include <memory>
#include <mutex>
#include <string>
#include <vector>

using namespace tc;

struct tc_stream {
    tc_ctx *ctx = nullptr;
    cudaStream_t st = nullptr;
    bool owned = false;
    void *ws = nullptr;              // repacked operands + split-K partials
    size_t ws_cap = 0;
    void *rx = nullptr;              // relaxed fp32: the bf16 split operands
    size_t rx_cap = 0;
    unsigned *status_host = nullptr; // mapped, pinned: kernels report timeouts here
    unsigned *status_dev = nullptr;
};

struct tc_ctx {
    int device = 0;
    int num_sms = 0;
    tc_stream *def = nullptr;
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    std::string last = "none";
    uint64_t launches = 0;
    void *dbuf[3] = {nullptr, nullptr, nullptr};  // device copies for tc_gemm_host
    size_t dcap[3] = {0, 0, 0};
    cudaStream_t copy_in = nullptr, copy_out = nullptr;   // tc_gemm_host's copy streams
    std::vector<cudaEvent_t> host_ev;              // tc_gemm_host's events, created once and reused
    std::mutex host_mu;                            // one tc_gemm_host at a time (it owns dbuf, host_ev)
    int max_pairs[3] = {-1, -1, -1};               // resident CTA pairs (BN 128, 192, 256), queried once
    int csplit_clusters[2][17];                    // resident cluster splits (BN 64, 128; S), -1 = not queried
    std::mutex mu;
    tc_ctx()
    {
        for (auto &row : csplit_clusters)
            for (int &v : row) v = -1;
    }
};

namespace {

size_t elem_size(tc_dtype_t t) { return t == TC_F32 ? 4 : t == TC_I8 ? 1 : 2; }

bool mul_ok(int64_t a, int64_t b, int64_t *out) { return !__builtin_mul_overflow(a, b, out); }
bool add_ok(int64_t a, int64_t b, int64_t *out) { return !__builtin_add_overflow(a, b, out); }

// A problem after validation: normalised leading dimensions and extents.
struct Norm {
    int64_t lda, ldb, ldc;
    int64_t a_rows, a_cols, b_rows, b_cols;   // stored shapes
    int64_t batch, sa, sb, sc;                // batch and element strides
    int64_t a_bytes, b_bytes, c_bytes;        // byte extents touched (all batch entries)
};

// Extent in elements of a stored rows x cols matrix with leading dim ld,
// repeated `batch` times at `stride`.
bool extent(int64_t rows, int64_t cols, int64_t ld, int64_t batch, int64_t stride, int64_t esz,
            int64_t *bytes)
{
    int64_t e, t;
    if (!mul_ok(rows - 1, ld, &e) || !add_ok(e, cols, &e)) return false;
    if (batch > 1) {
        if (!mul_ok(batch - 1, stride, &t) || !add_ok(e, t, &e)) return false;
    }
    return mul_ok(e, esz, bytes);
}

bool ranges_overlap(const void *p, int64_t pb, const void *q, int64_t qb)
{
    const uintptr_t a0 = (uintptr_t)p, a1 = a0 + (uintptr_t)pb;
    const uintptr_t b0 = (uintptr_t)q, b1 = b0 + (uintptr_t)qb;
    return a0 < b1 && b0 < a1;
}

// Operand types each entry point accepts: the GEMM (a == b in f16, bf16,
// f32), the integer GEMM (int8 x int8, int32 accumulation, fp32 C) and the
// int8-weight product (f16/bf16 activations, int8 weights stored [N,K]).
enum ValidateMode { V_GEMM = 0, V_I8 = 1, V_Q8W = 2 };

tc_status_t validate(const tc_gemm_desc *d, const void *A, const void *B, const void *C, int64_t batch,
                     int64_t sa, int64_t sb, int64_t sc, Norm *n, int mode = V_GEMM)
{
    if (!d || !A || !B || !C) return TC_ERR_NULL;
    if (d->M < 1 || d->N < 1 || d->K < 1 || batch < 1) return TC_ERR_DIM;
    if (mode == V_Q8W) {
        if ((d->a_dtype != TC_F16 && d->a_dtype != TC_BF16) || d->b_dtype != TC_I8 || d->accum_dtype != TC_F32 ||
            (d->c_dtype != d->a_dtype && d->c_dtype != TC_F32))
            return TC_ERR_DTYPE;
        if (d->transpose_a || !d->transpose_b) return TC_ERR_LAYOUT;
    } else if (d->a_dtype == TC_I8) {
        if (mode != V_I8 || d->b_dtype != TC_I8 || d->accum_dtype != TC_I32 || d->c_dtype != TC_F32)
            return TC_ERR_DTYPE;
    } else {
        const bool ab_ok = d->a_dtype == TC_F16 || d->a_dtype == TC_BF16 || d->a_dtype == TC_F32;
        if (!ab_ok || d->b_dtype != d->a_dtype || d->accum_dtype != TC_F32 ||
            (d->c_dtype != d->a_dtype && d->c_dtype != TC_F32))
            return TC_ERR_DTYPE;
    }
    if (d->lda < 0 || d->ldb < 0 || d->ldc < 0) return TC_ERR_LD;
    if (sa < 0 || sb < 0 || sc < 0) return TC_ERR_STRIDE;

    Norm r;
    r.a_rows = d->transpose_a ? d->K : d->M;
    r.a_cols = d->transpose_a ? d->M : d->K;
    r.b_rows = d->transpose_b ? d->N : d->K;
    r.b_cols = d->transpose_b ? d->K : d->N;
    r.lda = d->lda ? d->lda : r.a_cols;
    r.ldb = d->ldb ? d->ldb : r.b_cols;
    r.ldc = d->ldc ? d->ldc : d->N;
    if (r.lda < r.a_cols || r.ldb < r.b_cols || r.ldc < d->N) return TC_ERR_LD;
    r.batch = batch;
    r.sa = sa;
    r.sb = sb;
    r.sc = sc;
    const int64_t ea = (int64_t)elem_size(d->a_dtype), eb = (int64_t)elem_size(d->b_dtype),
                  ec = (int64_t)elem_size(d->c_dtype);
    if (!extent(r.a_rows, r.a_cols, r.lda, batch, sa, ea, &r.a_bytes) ||
        !extent(r.b_rows, r.b_cols, r.ldb, batch, sb, eb, &r.b_bytes) ||
        !extent(d->M, d->N, r.ldc, batch, sc, ec, &r.c_bytes))
        return TC_ERR_OVERFLOW;
    if (batch > 1) {
        // distinct batch entries must not write the same C elements
        int64_t c_one;
        if (!extent(d->M, d->N, r.ldc, 1, 0, 1, &c_one)) return TC_ERR_OVERFLOW;
        if (sc < c_one) return TC_ERR_STRIDE;
    }
    if (!std::isfinite(d->alpha) || !std::isfinite(d->beta)) return TC_ERR_SCALAR;
    if (ranges_overlap(C, r.c_bytes, A, r.a_bytes) || ranges_overlap(C, r.c_bytes, B, r.b_bytes))
        return TC_ERR_OVERLAP;
    *n = r;
    return TC_OK;
}

// --------------------------------------------------------------- dispatch

// int8 GEMM limits: K at most I8_K_MAX; K slices of I8_SLICE_KB blocks (1024
// products, |sum| <= 2^24: exact in an fp32 accumulator); the slices are
// summed on chip as int32 when K <= I8_ONCHIP_K_MAX (|sum| <= 2^14 K <= 2^30).
constexpr int I8_K_MAX = 131072;
constexpr int I8_SLICE_KB = 16;
constexpr int I8_ONCHIP_K_MAX = 65536;    // int32 running sums: |sum| <= 2^14 K <= 2^30

struct Plan {
    bool ffma = false;
    int ffma_tile = FFMA_SMALL;
    int bn = 256, cg = 1, split = 1, grid = 1, group_m = 8;
    bool i8acc = false;        // int8: exact K slices summed in TMEM (one unit per tile)
    bool csplit = false;       // split-K as clusters of K slices reduced on chip (seg0_split CTAs per cluster)
    // the skinny-product kernel (gemv.cu): X = op(A) and W = B (rows N), or,
    // when swapped, X = B^T (N rows) and W = A (rows M); K split over a
    // cluster of gemv_ks CTAs
    bool gemv = false, gemv_swap = false;
    int gemv_ks = 1;
    int64_t seg0_tiles = 0, split_base = 0;
    int seg0_split = 1, seg1_split = 1;
    bool tma_store = true;
    bool pack_a = false, pack_b = false;
    int64_t tiles = 0, units = 0;
    std::string name;
};

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// Environment override for tests and sweeps: TC_FORCE_VARIANT holds
// space/comma separated tokens: bn=<64|128|192|256> split=<S> grid=<G>
// group_m=<G> ffma=<small|large|panel> pack=<1> tail=<S> (K slices of the
// last-wave tiles; 0 or 1 disables) sms=<N> (plan for N SMs) cg=<1|2>
// (CTAs per tile) store=direct (plain stores of C instead of TMA stores)
// grouped=0 (a grouped call enqueues its problems one by one) chunk=0 (an
// MN-major operand is read 64 columns per copy instead of one chunked copy)
// i8acc=0 (int8: K slices through memory and the reduction kernel, not
// summed on chip) shorta=0 (a one-CTA tile copies all 128 rows of A even
// when A has fewer) csplit=0 (split-K slices go through global memory and
// the reduction kernel instead of a cluster reduction on chip) gemv=0 (a
// product with at most 16 rows on one side stays on the tensor-core kernel)
// gemv_ks=<1|2|4|8> (the skinny-product kernel's cluster form with this K
// split) gemv_rr=0 (its cluster form instead of the row-range form)
// gemv_blocks=0|1 (the row-range form on 2 CTAs per SM, sharing rows or
// whole 16-row blocks) gemv_grid=<G> (the row-range form on G CTAs)
// hband=<rows> (tc_gemm_host moves A and C in bands of this many rows).
// Test hooks: debug_drop=1 (the MMA warp withholds the first tile's
// "accumulator ready" signal, so the epilogue's wait expires) and
// debug_timeout_ms=<ms> (the bound on every device wait).
struct Force {
    int bn = 0, split = 0, grid = 0, group_m = 0, ffma = -1, pack = 0, tail = -1, sms = 0, cg = 0;
    bool direct_store = false;
    int grouped = 1;
    int debug_drop = 0, debug_timeout_ms = 0;
    int no_chunk = 0;
    int no_short_a = 0;
    int host_band = 0;
    int i8acc = -1;
    int csplit = -1;
    int gemv = -1, gemv_ks = 0, gemv_rr = -1, gemv_blocks = -1, gemv_grid = 0;
};

Force read_force()
{
    Force f;
    const char *e = std::getenv("TC_FORCE_VARIANT");
    if (!e) return f;
    std::string s(e);
    for (auto &ch : s)
        if (ch == ',') ch = ' ';
    size_t pos = 0;
    while (pos < s.size()) {
        size_t end = s.find(' ', pos);
        if (end == std::string::npos) end = s.size();
        std::string tok = s.substr(pos, end - pos);
        pos = end + 1;
        const size_t eq = tok.find('=');
        if (eq == std::string::npos) continue;
        const std::string k = tok.substr(0, eq), v = tok.substr(eq + 1);
        if (k == "bn") f.bn = std::atoi(v.c_str());
        else if (k == "split") f.split = std::atoi(v.c_str());
        else if (k == "grid") f.grid = std::atoi(v.c_str());
        else if (k == "group_m") f.group_m = std::atoi(v.c_str());
        else if (k == "ffma") f.ffma = (v == "large") ? FFMA_LARGE : (v == "panel") ? FFMA_PANEL : FFMA_SMALL;
        else if (k == "pack") f.pack = std::atoi(v.c_str());
        else if (k == "tail") f.tail = std::atoi(v.c_str());
        else if (k == "sms") f.sms = std::atoi(v.c_str());
        else if (k == "cg") f.cg = std::atoi(v.c_str());
        else if (k == "store") f.direct_store = (v == "direct");
        else if (k == "grouped") f.grouped = std::atoi(v.c_str());
        else if (k == "debug_drop") f.debug_drop = std::atoi(v.c_str());
        else if (k == "debug_timeout_ms") f.debug_timeout_ms = std::atoi(v.c_str());
        else if (k == "chunk") f.no_chunk = std::atoi(v.c_str()) == 0;
        else if (k == "shorta") f.no_short_a = std::atoi(v.c_str()) == 0;
        else if (k == "hband") f.host_band = std::atoi(v.c_str());
        else if (k == "i8acc") f.i8acc = std::atoi(v.c_str());
        else if (k == "csplit") f.csplit = std::atoi(v.c_str());
        else if (k == "gemv") f.gemv = std::atoi(v.c_str());
        else if (k == "gemv_ks") f.gemv_ks = std::atoi(v.c_str());
        else if (k == "gemv_rr") f.gemv_rr = std::atoi(v.c_str());
        else if (k == "gemv_blocks") f.gemv_blocks = std::atoi(v.c_str());
        else if (k == "gemv_grid") f.gemv_grid = std::atoi(v.c_str());
    }
    return f;
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Relative main-loop throughput per SM of each kernel shape (CTAs per tile,
// tile width), measured on GB300 with bf16 at M = N = 4096 and long K:
// narrower tiles read more shared memory per MMA flop, and a CTA pair
// (tcgen05.mma.cta_group::2) loads half of B per SM.  The 256 x 192 pair
// measured the same per SM as the one-CTA 128 x 192 tile (fp16 8192 x 384
// x 4096: 30.9 us both); on a tie the pair, listed first, is taken (it
// reads B from L2 half as often).
double tile_rate(int cg, int bn)
{
    if (cg == 2) return bn == 256 ? 1.15 : bn == 192 ? 0.87 : 0.72;
    return bn == 256 ? 1.0 : bn == 192 ? 0.87 : bn == 128 ? 0.63 : 0.45;
}

// Modelled fixed cost of a split-K reduction (its launch, the wait for the
// GEMM grid, one pass over the partial tiles), in the schedule's time unit:
// one K block of one 256-wide tile column at tile rate 1, ~1 ns on GB300.
constexpr double SPLIT_FIXED = 4500.0;
// The same for a cluster split (two cluster barriers and one pass over the
// slices' shared memory, inside the GEMM kernel).
constexpr double CSPLIT_FIXED = 1200.0;
constexpr int CSPLIT_MAX = 16;      // CTAs per cluster (non-portable size)

// Persistent schedule of `tiles` output tiles on num_sms CTAs: whole waves
// of tiles, then the partial last wave.  When the last wave leaves at least
// half of the SMs idle, its tiles are cut into K slices (reduced in fixed
// order) so that every SM gets work.
struct Sched {
    int64_t tiles, seg0_tiles;
    int seg0_split, seg1_split;
    double t;   // modelled time, in units of one BN=256 tile
};

Sched schedule(int64_t tiles, int64_t num_kb, int num_sms, int cg, int bn, int force_tail)
{
    const int64_t G = std::min<int64_t>(tiles, num_sms);
    const int64_t full = tiles / G, L = tiles % G;
    Sched s{tiles, tiles, 1, 1, 0.0};
    if (L > 0 && full >= 1) {
        int64_t S2 = std::min<int64_t>(std::min<int64_t>(G / L, num_kb / 4), 4);
        if (force_tail >= 0) S2 = force_tail;
        if (S2 >= 2) {
            s.seg0_tiles = tiles - L;
            s.seg1_split = (int)S2;
        }
    }
    const double tail = L == 0 ? 0.0 : (s.seg1_split > 1 ? 1.0 / s.seg1_split + 0.05 : 1.0);
    s.t = ((double)full + tail) * bn / tile_rate(cg, bn);
    return s;
}

int pow2_floor(int x)
{
    int p = 1;
    while (p * 2 <= x) p *= 2;
    return p;
}

// K split of the skinny-product kernel: clusters of up to 8 CTAs along K
// until there are at least two CTAs per SM, keeping at least 32 K steps
// (4 per warp) per CTA.
int gemv_ksplit(int64_t rows_w, int64_t K, bool w_i8, int num_sms)
{
    const int64_t blocks = cdiv(rows_w, 16);
    const int64_t steps = cdiv(K, w_i8 ? 64 : 32);
    int ks = 1;
    while (ks < 8 && blocks * ks < 2LL * num_sms && steps / (2LL * ks) >= 32) ks *= 2;
    return ks;
}

// The row-range form of the skinny-product kernel applies when every row of
// X and W starts on a 16-byte boundary and there are at least as many W rows
// as SMs: two persistent CTAs per SM (fewer when rows are few), each owning
// an equal share of the rows. Where W has more 16-row blocks than CTAs, the shares are whole blocks on
// as few CTAs as keep the passes per CTA at their least (x[4,4096]
// W[11008,4096]: 688 blocks, 230 CTAs of 3 blocks, 20.1 us, against 304 CTAs
// of 36.2 rows each -- three passes, the last a quarter full -- 21.8 us).
bool plan_gemv_rr(GemvArgs &g, int num_sms)
{
    if (!g.x_vec || !g.w_vec || g.rows_w < num_sms) return false;
    g.rowrange = 1;
    const int64_t nb = cdiv(g.rows_w, 16), ctas = 2LL * num_sms;
    g.block_rows = nb > ctas;
    g.grid = (int)(g.block_rows ? cdiv(nb, cdiv(nb, ctas)) : std::min<int64_t>(ctas, g.rows_w));
    return true;
}

// allow_gemv: the call may take the skinny-product kernel (a plain GEMM:
// no fused epilogue, no per-column scale).
tc_status_t make_plan(const tc_gemm_desc *d, const Norm &n, const void *A, const void *B, int num_sms,
                      Plan *out, bool allow_gemv = true)
{
    Plan p;
    const Force f = read_force();
    if (f.sms > 0) num_sms = f.sms;
    if (num_sms < 1) num_sms = 1;
    const char *lay = d->transpose_a ? (d->transpose_b ? "tt" : "tn") : (d->transpose_b ? "nt" : "nn");
    const char *dt = d->a_dtype == TC_F32 ? "f32" : d->a_dtype == TC_BF16 ? "bf16" : "f16";
    const char *ct = d->c_dtype == TC_F32 ? "f32" : d->c_dtype == TC_BF16 ? "bf16" : "f16";
    char buf[160];

    if (d->a_dtype == TC_F32) {
        // fp32-exact path on CUDA cores: 128x128 tiles when they fill the
        // SMs, whole-K panels of 16x32 tiles for small outputs, else 32x32
        p.ffma = true;
        const int64_t big_tiles = cdiv(d->M, 128) * cdiv(d->N, 128) * n.batch;
        const int64_t panel_tiles = cdiv(d->M, 16) * cdiv(d->N, 32) * n.batch;
        p.ffma_tile = big_tiles >= num_sms ? FFMA_LARGE : panel_tiles <= 8 * num_sms ? FFMA_PANEL : FFMA_SMALL;
        if (f.ffma >= 0) p.ffma_tile = f.ffma;
        std::snprintf(buf, sizeof buf, "ffma_f32_%s_%s", lay,
                      p.ffma_tile == FFMA_LARGE ? "128x128" : p.ffma_tile == FFMA_PANEL ? "16x32_panel" : "32x32");
        p.name = buf;
        *out = p;
        return TC_OK;
    }

    // At most GEMV_MAX_ROWS rows on one side of an NT product (both operands
    // K-contiguous: the decode shape x[M, K] @ W[N, K]^T): the weight side is
    // streamed once by the skinny-product kernel instead of padding a
    // 128-row tensor-core tile.
    if (allow_gemv && f.gemv != 0 && n.batch == 1 && !d->transpose_a && d->transpose_b &&
        (d->M <= GEMV_MAX_ROWS || d->N <= GEMV_MAX_ROWS)) {
        p.gemv = true;
        p.gemv_swap = d->M > GEMV_MAX_ROWS;
        const int64_t rows_w = p.gemv_swap ? d->M : d->N, rows_x = p.gemv_swap ? d->N : d->M;
        p.gemv_ks = f.gemv_ks > 0 ? pow2_floor(std::min(f.gemv_ks, 8)) : gemv_ksplit(rows_w, d->K, false, num_sms);
        std::snprintf(buf, sizeof buf, "gemv_%s_%s_%s_x%d%s", lay, dt, ct, (int)rows_x, p.gemv_swap ? "_swap" : "");
        p.name = buf;
        *out = p;
        return TC_OK;
    }

    // TMA reads an operand in place only with a 16-byte aligned base and
    // 16-byte multiple row (and batch) strides; otherwise it is repacked.
    const bool a3 = n.batch > 1 && n.sa != 0, b3 = n.batch > 1 && n.sb != 0;
    p.pack_a = !aligned16(A) || (n.lda % 8) != 0 || (a3 && (n.sa % 8) != 0);
    p.pack_b = !aligned16(B) || (n.ldb % 8) != 0 || (b3 && (n.sb % 8) != 0);
    if (f.pack) p.pack_a = p.pack_b = true;

    const int64_t num_kb = cdiv(d->K, BK);
    const int64_t tiles128 = cdiv(d->M, BM) * cdiv(d->N, 128) * n.batch;
    int bn = 0, cg = 1;
    Sched sc{};
    bool split_k = (f.split == 0 && f.cg != 2 && tiles128 * 2 <= num_sms && num_kb >= 16) || f.split > 0;
    // cluster split (slices reduced on chip in one launch) unless disabled or
    // a forced split is longer than a cluster can be
    const bool csplit_ok = f.csplit != 0 && f.cg != 2 && (f.split == 0 || f.split <= CSPLIT_MAX);
    if (split_k && f.split == 0 && f.bn == 0) {
        // 64-wide whole-K tiles instead, when they fill at least half the SMs
        // and the split's reduction would cost more than their lower rate
        // (e.g. fp16 1024^3 on GB300: 13.8 us against 16.7 us split in two
        // through memory)
        const int64_t tiles64 = cdiv(d->M, BM) * cdiv(d->N, 64) * n.batch;
        const int64_t split = std::min<int64_t>(std::max<int64_t>(num_sms / tiles128, 1), num_kb / 4);
        const double t_split = (double)cdiv(num_kb, split) * 128.0 / tile_rate(1, 128) +
                               (csplit_ok ? CSPLIT_FIXED : SPLIT_FIXED);
        const double t_64 = (double)cdiv(tiles64, num_sms) * (double)num_kb * 64.0 / tile_rate(1, 64);
        if (tiles64 * 2 >= num_sms && t_64 < t_split) {
            split_k = false;
            bn = 64;
            sc = schedule(tiles64, num_kb, num_sms, 1, 64, f.tail);
        }
    }
    if (split_k) {
        // split-K: too few output tiles to occupy the SMs and a long K loop
        bn = f.bn ? f.bn : 128;
        int64_t tiles = cdiv(d->M, BM) * cdiv(d->N, bn) * n.batch;
        int split = f.split > 0 ? f.split
                                : (int)std::min<int64_t>(std::max<int64_t>(num_sms / tiles, 1), num_kb / 4);
        split = (int)std::min<int64_t>(std::max(split, 1), num_kb);
        if (csplit_ok && (bn == 64 || bn == 128)) {
            // Cluster split: at most CSPLIT_MAX slices per tile.  Tile width
            // 128 or 64, whichever leaves each CTA fewer operand bytes to
            // load (per CTA: ceil(K blocks / S) stages, times the waves of
            // clusters), since these shapes are bound by how fast each CTA
            // pulls its operands, not by the tensor core.
            int best_bn = 0, best_s = 0;
            double best_cost = 1e300;
            for (int b : {128, 64}) {
                if (f.bn && b != f.bn) continue;
                const int64_t t = cdiv(d->M, BM) * cdiv(d->N, b) * n.batch;
                int64_t S = f.split > 0 ? f.split
                                        : std::min<int64_t>({(int64_t)CSPLIT_MAX, std::max<int64_t>(num_sms / t, 1),
                                                             num_kb / 4});
                S = std::min<int64_t>(S, num_kb);
                if (S < 2) continue;
                const double waves = std::ceil((double)(t * S) / num_sms);
                const double cost = waves * (double)cdiv(num_kb, S) * (double)stage_bytes(b, 1);
                if (cost < best_cost - 1e-9) {
                    best_cost = cost;
                    best_bn = b;
                    best_s = (int)S;
                }
            }
            if (best_bn) {
                p.csplit = true;
                bn = best_bn;
                split = best_s;
                tiles = cdiv(d->M, BM) * cdiv(d->N, bn) * n.batch;
            }
        }
        sc = {tiles, tiles, split, 1, 0.0};
    } else if (bn == 64) {
        cg = 1;
    } else {
        // the kernel shape (CTAs per tile, tile width) with the least modelled time
        static const int shapes[][2] = {{2, 256}, {1, 256}, {2, 192}, {1, 192}, {2, 128}, {1, 128}, {1, 64}};
        double best = 1e300;
        for (const auto &sh : shapes) {
            const int c = sh[0], b = sh[1];
            if (f.cg && c != f.cg) continue;
            if (f.bn ? b != f.bn : b == 64) continue;      // 64-wide tiles only on request
            const int workers = c == 2 ? std::max(num_sms / 2, 1) : num_sms;
            const Sched t = schedule(cdiv(d->M, BM * c) * cdiv(d->N, b) * n.batch, num_kb, workers, c, b, f.tail);
            if (t.t < best - 1e-9) {
                best = t.t;
                bn = b;
                cg = c;
                sc = t;
            }
        }
        // A short K loop (under 16 blocks) on one wave of tiles: a tile's
        // fixed costs -- set-up, the first loads' latency, the epilogue of
        // its 128 x BN/CG outputs -- outweigh the rates above, and a tile of
        // any width up to 256 takes the same MMA time (the ~128-cycle
        // tcgen05.mma floor).  So 128 x 64 one-CTA tiles when they fit in
        // one wave (fp16 512^3: 6.7 us against 8.3 with 256 x 128 pairs;
        // 256^3: 5.8 against 7.1), else one-CTA tiles of the chosen width
        // when those do (bf16 2048 x 2048 x 512: 9.9 against 10.2 us).
        if (!f.cg && !f.bn && num_kb < 16) {
            const int64_t tiles64 = cdiv(d->M, BM) * cdiv(d->N, 64) * n.batch;
            const int64_t tiles1 = cdiv(d->M, BM) * cdiv(d->N, bn) * n.batch;
            if (tiles64 <= num_sms) {
                bn = 64;
                cg = 1;
                sc = schedule(tiles64, num_kb, num_sms, 1, 64, f.tail);
            } else if (cg == 2 && tiles1 <= num_sms) {
                cg = 1;
                sc = schedule(tiles1, num_kb, num_sms, 1, bn, f.tail);
            }
        }
    }
    const int workers = cg == 2 ? std::max(num_sms / 2, 1) : num_sms;   // tiles in flight
    if (bn == 0) return TC_ERR_VARIANT;
    p.bn = bn;
    p.cg = cg;
    p.tiles = sc.tiles;
    p.seg0_tiles = sc.seg0_tiles;
    p.seg0_split = sc.seg0_split;
    p.seg1_split = sc.seg1_split;
    p.units = sc.seg0_tiles * sc.seg0_split + (sc.tiles - sc.seg0_tiles) * sc.seg1_split;
    p.split_base = sc.seg0_split > 1 ? 0 : sc.seg0_tiles;
    p.split = (sc.seg0_split > 1 || (sc.tiles > sc.seg0_tiles && sc.seg1_split > 1)) ? 2 : 1;
    if (p.units > INT32_MAX / 2) return TC_ERR_OVERFLOW;
    p.grid = (int)std::min<int64_t>(p.units, workers);
    if (f.grid > 0) p.grid = (int)std::min<int64_t>(f.grid, p.units);
    if (p.csplit) p.grid = (int)p.units;           // one CTA per (tile, slice): clusters of slices
    p.grid *= cg;                                  // CTAs
    p.group_m = f.group_m > 0 ? f.group_m : 4;
    p.tma_store = !f.direct_store;
    std::snprintf(buf, sizeof buf, "tcgen05_%s_%s_%s_%dx%d%s%s%s%s", lay, dt, ct, BM * cg, bn,
                  cg == 2 ? "_pair" : "", sc.seg0_split > 1 ? (p.csplit ? "_csplit" : "_splitk") : "",
                  p.pack_a ? "_packA" : "",
                  p.pack_b ? "_packB" : "");
    p.name = buf;
    if (sc.seg0_split > 1) {
        std::snprintf(buf, sizeof buf, "_s%d", sc.seg0_split);
        p.name += buf;
    } else if (sc.tiles > sc.seg0_tiles) {
        std::snprintf(buf, sizeof buf, "_tail%dx%d", (int)(sc.tiles - sc.seg0_tiles), sc.seg1_split);
        p.name += buf;
    }
    *out = p;
    return TC_OK;
}

// --------------------------------------------------------------- resources

tc_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? TC_OK : TC_ERR_CUDA; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

tc_status_t ensure_ws(tc_stream *s, size_t bytes)
{
    if (bytes <= s->ws_cap) return TC_OK;
    size_t cap = round_up(bytes + bytes / 4, (size_t)1 << 20);
    if (s->ws) {
        cudaError_t e = cudaFreeAsync(s->ws, s->st);
        s->ws = nullptr;
        s->ws_cap = 0;
        if (e != cudaSuccess) return TC_ERR_CUDA;
    }
    if (cudaMallocAsync(&s->ws, cap, s->st) != cudaSuccess) {
        s->ws = nullptr;
        return TC_ERR_CUDA;
    }
    s->ws_cap = cap;
    return TC_OK;
}

bool encode_map(tc_ctx *ctx, CUtensorMap *m, tc_dtype_t dt, const void *base, int64_t inner, int64_t outer,
                int64_t ld_elems, bool three_d, int64_t batch, int64_t bstride_elems, uint32_t box_inner,
                uint32_t box_outer, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B)
{
    const CUtensorMapDataType t = dt == TC_BF16  ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                  : dt == TC_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const int64_t es = (int64_t)elem_size(dt);
    cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)outer, (cuuint64_t)batch};
    cuuint64_t strides[2] = {(cuuint64_t)(ld_elems * es), (cuuint64_t)(bstride_elems * es)};
    cuuint32_t box[3] = {box_inner, box_outer, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = ctx->encode(m, t, three_d ? 3 : 2, const_cast<void *>(base), dims, strides, box, estr,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// An MN-major operand (K rows of `extent` elements, leading dimension ld)
// viewed as 64-element rows x K x extent/64 chunks, so that one box of
// {64, 64, chunks} brings `chunks` adjacent 64-wide slices of one K block,
// each as a 64 x 64 swizzled tile 8 KB after the previous one -- the layout
// that separate 64-wide boxes give.  Only for extents that are multiples of
// 64: no chunk then reaches past a row's last element.
// With width 32 the chunks are 32 elements (64 bytes) with the 64-byte
// swizzle, 4 KB apart: the layout of a B share that is not a multiple of
// 64 columns.
bool encode_chunked(tc_ctx *ctx, CUtensorMap *m, tc_dtype_t dt, const void *base, int64_t extent, int64_t k,
                    int64_t ld_elems, uint32_t chunks, uint32_t width = 64)
{
    if (extent % width != 0) return false;
    const CUtensorMapDataType t = dt == TC_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const int64_t es = 2;
    cuuint64_t dims[3] = {width, (cuuint64_t)k, (cuuint64_t)(extent / width)};
    cuuint64_t strides[2] = {(cuuint64_t)(ld_elems * es), (cuuint64_t)(width * es)};
    cuuint32_t box[3] = {width, 64, chunks};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = ctx->encode(m, t, 3, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                             width == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

tc_status_t read_status(tc_stream *s)
{
    volatile unsigned *st = s->status_host;
    if (st && *st != 0u) {
        *st = 0u;
        return TC_ERR_DEVICE_TIMEOUT;
    }
    return TC_OK;
}

// Enqueue one validated, planned problem on stream s (epi: the fused
// bias/activation epilogue, or null).
// col_scale: the int8 path's per-column dequantisation (its K slices then
// hold integers and are added as such), or null.
// Launch the skinny-product kernel on stream s: the row-range form when it
// applies (and no K split was forced), else the cluster form.
tc_status_t enqueue_gemv(tc_ctx *ctx, tc_stream *s, GemvArgs &g, const Force &f, std::string &name)
{
    char buf[48];
    if (f.gemv_rr != 0 && f.gemv_ks == 0 && plan_gemv_rr(g, ctx->num_sms)) {
        if (f.gemv_blocks >= 0 && f.gemv_blocks != g.block_rows) {
            g.block_rows = f.gemv_blocks != 0;
            g.grid = (int)std::min<int64_t>(2LL * ctx->num_sms, g.rows_w);
        }
        if (f.gemv_grid > 0) g.grid = (int)std::min<int64_t>(f.gemv_grid, g.rows_w);
        std::snprintf(buf, sizeof buf, "_rr%d%s", g.grid, g.block_rows ? "b" : "");
    } else {
        g.rowrange = 0;
        std::snprintf(buf, sizeof buf, "_ks%d", g.ksplit);
    }
    if (launch_gemv(g, s->st) != cudaSuccess) return TC_ERR_CUDA;
    ctx->launches += 1;
    name += buf;
    return TC_OK;
}

// int_slices: the int8 path -- K slices hold exact integers and are added
// as integers (through memory only, never a cluster split).
tc_status_t enqueue(tc_ctx *ctx, const tc_gemm_desc *d, const Norm &n, const Plan &plan, const void *A,
                    const void *B, void *C, tc_stream *s, const tc_epilogue *epi = nullptr,
                    const float *col_scale = nullptr, bool int_slices = false)
{
    cudaError_t e;
    Plan p = plan;
    if (p.gemv) {
        GemvArgs g{};
        g.X = p.gemv_swap ? B : A;
        g.W = p.gemv_swap ? A : B;
        g.C = C;
        g.scale = nullptr;
        g.rows_x = p.gemv_swap ? d->N : d->M;
        g.rows_w = p.gemv_swap ? d->M : d->N;
        g.K = d->K;
        g.ldx = p.gemv_swap ? n.ldb : n.lda;
        g.ldw = p.gemv_swap ? n.lda : n.ldb;
        g.c_sx = p.gemv_swap ? 1 : n.ldc;
        g.c_sw = p.gemv_swap ? n.ldc : 1;
        g.c_dtype = d->c_dtype;
        g.alpha = d->alpha;
        g.beta = d->beta;
        g.x_vec = aligned16(g.X) && (g.ldx * 2) % 16 == 0;
        g.w_vec = aligned16(g.W) && (g.ldw * 2) % 16 == 0;
        g.w_i8 = 0;
        g.x_bf16 = d->a_dtype == TC_BF16;
        g.ksplit = p.gemv_ks;
        std::string name = p.name;
        const tc_status_t st = enqueue_gemv(ctx, s, g, read_force(), name);
        if (st != TC_OK) return st;
        ctx->last = name;
        return TC_OK;
    }
    if (p.csplit) {
        // A cluster split needs its clusters of K slices to be schedulable
        // on this device, and all of them resident at once: a second wave
        // of clusters doubles the time (on GB300 only 7 clusters of 16 fit,
        // 8 of 12).  Unless the split was forced, the slice count shrinks
        // until every tile's cluster is resident; with no schedulable
        // cluster at all the same slices go through global memory.
        auto clusters = [&](int S) {
            int &mc = ctx->csplit_clusters[p.bn == 64 ? 0 : 1][std::min(S, CSPLIT_MAX)];
            if (mc < 0) mc = max_active_csplit_clusters(p.bn, S);
            return mc;
        };
        int S = p.seg0_split;
        if (read_force().split == 0)
            while (S > 2 && clusters(S) < p.tiles) --S;
        if (clusters(S) < 1 || int_slices) {
            p.csplit = false;
            p.grid = (int)std::min<int64_t>(p.units, ctx->num_sms);
            const std::string::size_type at = p.name.find("_csplit");
            if (at != std::string::npos) p.name.replace(at, 7, "_splitk");
        } else if (S != p.seg0_split) {
            p.seg0_split = S;
            p.units = p.tiles * S;
            p.grid = (int)p.units;
            p.name = p.name.substr(0, p.name.rfind("_s")) + "_s" + std::to_string(S);
        }
    }
    if (p.ffma) {
        FfmaArgs a{};
        a.M = d->M;
        a.N = d->N;
        a.K = d->K;
        a.batch = (int)n.batch;
        a.ta = d->transpose_a;
        a.tb = d->transpose_b;
        a.A = static_cast<const float *>(A);
        a.B = static_cast<const float *>(B);
        a.C = static_cast<float *>(C);
        a.lda = n.lda;
        a.ldb = n.ldb;
        a.ldc = n.ldc;
        a.stride_a = n.sa;
        a.stride_b = n.sb;
        a.stride_c = n.sc;
        a.alpha = d->alpha;
        a.beta = d->beta;
        e = launch_ffma(a, p.ffma_tile, s->st);
        if (e != cudaSuccess) return TC_ERR_CUDA;
        ctx->launches += 1;
        ctx->last = p.name;
        return TC_OK;
    }

    // ---- workspace: [packed A | packed B | split-K partials]
    const int64_t a_batch = (n.batch > 1 && n.sa != 0) ? n.batch : 1;
    const int64_t b_batch = (n.batch > 1 && n.sb != 0) ? n.batch : 1;
    // repacked rows padded to 64 elements: 128-byte aligned rows for TMA
    const int64_t lda_p = p.pack_a ? (int64_t)round_up((size_t)n.a_cols, 64) : n.lda;
    const int64_t ldb_p = p.pack_b ? (int64_t)round_up((size_t)n.b_cols, 64) : n.ldb;
    const size_t a_pack_bytes = p.pack_a ? round_up((size_t)(n.a_rows * lda_p * a_batch * 2), 256) : 0;
    const size_t b_pack_bytes = p.pack_b ? round_up((size_t)(n.b_rows * ldb_p * b_batch * 2), 256) : 0;
    const bool partials = p.split > 1 && !p.csplit;     // K slices summed through global memory
    const size_t part_bytes =
        partials ? (size_t)(p.units - p.split_base) * BM * p.cg * p.bn * sizeof(float) : 0;
    tc_status_t st = ensure_ws(s, a_pack_bytes + b_pack_bytes + part_bytes + 256);
    if (st != TC_OK) return st;
    uint8_t *ws = static_cast<uint8_t *>(s->ws);
    const void *Ause = A, *Buse = B;
    int64_t sa = n.sa, sb = n.sb;
    uint64_t launches = 0;
    PackBatch pb;
    pb.count = 0;
    if (p.pack_a) {
        pb.seg[pb.count++] = PackArgs{static_cast<const uint16_t *>(A), reinterpret_cast<uint16_t *>(ws), n.a_rows,
                                      n.a_cols, n.lda, lda_p, a_batch > 1 ? n.sa : 0, n.a_rows * lda_p, (int)a_batch};
        Ause = ws;
        sa = a_batch > 1 ? n.a_rows * lda_p : 0;
    }
    if (p.pack_b) {
        uint8_t *dst = ws + a_pack_bytes;
        pb.seg[pb.count++] = PackArgs{static_cast<const uint16_t *>(B), reinterpret_cast<uint16_t *>(dst), n.b_rows,
                                      n.b_cols, n.ldb, ldb_p, b_batch > 1 ? n.sb : 0, n.b_rows * ldb_p, (int)b_batch};
        Buse = dst;
        sb = b_batch > 1 ? n.b_rows * ldb_p : 0;
    }
    if (pb.count > 0) {
        if ((e = launch_pack(pb, s->st)) != cudaSuccess) return TC_ERR_CUDA;
        ++launches;
    }

    MmaLaunch L{};
    L.bn = p.bn;
    L.cg = p.cg;
    L.i8acc = p.i8acc ? 1 : 0;
    L.csplit = p.csplit ? 1 : 0;
    L.grid = p.grid;
    if (p.cg == 2) {
        // no more pairs than can be resident at once (a persistent grid)
        int &pairs = ctx->max_pairs[p.bn == 256 ? 2 : p.bn == 192 ? 1 : 0];
        if (pairs < 0) pairs = max_active_pairs(p.bn);
        if (pairs < 1) return TC_ERR_VARIANT;
        L.grid = std::min(L.grid, 2 * pairs);
    }
    MmaArgs &a = L.args;
    a.M = d->M;
    a.N = d->N;
    a.K = d->K;
    a.num_kb = (int)cdiv(d->K, BK);
    a.tiles_m = (int)cdiv(d->M, BM * p.cg);
    a.tiles_n = (int)cdiv(d->N, p.bn);
    a.tiles_per_batch = a.tiles_m * a.tiles_n;
    a.batch = (int)n.batch;
    a.seg0_tiles = (int)p.seg0_tiles;
    a.seg0_split = p.seg0_split;
    a.seg1_split = p.seg1_split;
    a.split_base = (int)p.split_base;
    a.total_units = (int)p.units;
    a.group_m = p.group_m;
    a.a_kmajor = !d->transpose_a;
    a.b_kmajor = d->transpose_b;
    a.a_3d = a_batch > 1;
    a.b_3d = b_batch > 1;
    // instruction descriptor (kind::f16): D f32 (bit 4), A/B format
    // (bits 7-9 / 10-12: 0 = f16, 1 = bf16), A/B MN-major (bits 15 / 16),
    // N >> 3 (bits 17-22), M >> 4 (bits 24-28)
    const uint32_t fmt = d->a_dtype == TC_BF16 ? 1u : 0u;
    a.idesc = (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(!a.a_kmajor) << 15) |
              ((uint32_t)(!a.b_kmajor) << 16) | ((uint32_t)(p.bn >> 3) << 17) |
              ((uint32_t)((BM * p.cg) >> 4) << 24);
    a.alpha = d->alpha;
    a.beta = d->beta;
    a.C = C;
    a.ldc = n.ldc;
    a.stride_c = n.batch > 1 ? n.sc : 0;
    a.c_dtype = d->c_dtype;
    const int64_t ec = (int64_t)elem_size(d->c_dtype);
    a.c_vec_ok = aligned16(C) && (n.ldc * ec) % 16 == 0 && (a.stride_c * ec) % 16 == 0;
    // C written through TMA stores of 32 x 32 chunks when its layout allows
    a.c_tma = a.c_vec_ok && p.tma_store;
    a.c_3d = n.batch > 1;
    a.ws = partials ? reinterpret_cast<float *>(ws + a_pack_bytes + b_pack_bytes) : nullptr;
    a.status = s->status_dev;
    a.bias = epi ? epi->bias : nullptr;
    a.act = epi ? (int)epi->activation : (int)TC_ACT_NONE;
    a.col_scale = col_scale;
    a.slice_kb = p.i8acc ? I8_SLICE_KB : 0;
    const int64_t kb_per_unit = a.num_kb;
    a.timeout_ns = 4000000000ull + (unsigned long long)kb_per_unit * 20000ull;
    {
        const Force f = read_force();
        if (f.debug_timeout_ms > 0) a.timeout_ns = (unsigned long long)f.debug_timeout_ms * 1000000ull;
        a.debug_drop_tfull = f.debug_drop;
    }

    const int64_t lda_use = p.pack_a ? lda_p : n.lda;
    const int64_t ldb_use = p.pack_b ? ldb_p : n.ldb;
    const bool chunk_ok = !read_force().no_chunk;
    bool ok;
    if (a.a_kmajor) {
        // a one-CTA tile taller than A: copy only A's rows (rounded up to 8)
        const uint32_t rows = (p.cg == 1 && d->M < BM && !read_force().no_short_a)
                                  ? (uint32_t)round_up((size_t)d->M, 8)
                                  : (uint32_t)BM;
        a.a_short_bytes = (int)((BM - rows) * BK * 2);
        ok = encode_map(ctx, &L.tmA, d->a_dtype, Ause, d->K, d->M, lda_use, a.a_3d, n.batch, sa, 64, rows);
    } else {
        a.a_chunked = chunk_ok && !a.a_3d && encode_chunked(ctx, &L.tmA, d->a_dtype, Ause, d->M, d->K, lda_use, BM / 64);
        ok = a.a_chunked || encode_map(ctx, &L.tmA, d->a_dtype, Ause, d->M, d->K, lda_use, a.a_3d, n.batch, sa, 64, 64);
    }
    if (ok) {
        if (a.b_kmajor) {
            ok = encode_map(ctx, &L.tmB, d->a_dtype, Buse, d->K, d->N, ldb_use, a.b_3d, n.batch, sb, 64,
                            (uint32_t)(p.bn / p.cg));
        } else if ((p.bn / p.cg) % 64 != 0) {
            // a share of 32-column chunks (64-byte swizzle), as the kernel expects
            a.b_chunked = chunk_ok && !a.b_3d &&
                          encode_chunked(ctx, &L.tmB, d->a_dtype, Buse, d->N, d->K, ldb_use,
                                         (uint32_t)(p.bn / p.cg / 32), 32);
            ok = a.b_chunked || encode_map(ctx, &L.tmB, d->a_dtype, Buse, d->N, d->K, ldb_use, a.b_3d, n.batch,
                                           sb, 32, 64, CU_TENSOR_MAP_SWIZZLE_64B);
        } else {
            a.b_chunked = chunk_ok && !a.b_3d &&
                          encode_chunked(ctx, &L.tmB, d->a_dtype, Buse, d->N, d->K, ldb_use,
                                         (uint32_t)(p.bn / p.cg / 64));
            ok = a.b_chunked ||
                 encode_map(ctx, &L.tmB, d->a_dtype, Buse, d->N, d->K, ldb_use, a.b_3d, n.batch, sb, 64, 64);
        }
    }
    if (ok && a.c_tma)
        ok = encode_map(ctx, &L.tmC, d->c_dtype, C, d->N, d->M, n.ldc, a.c_3d, n.batch, a.stride_c, 32, 32,
                        d->c_dtype == TC_F32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
    // split-K workspace: one row-major fp32 (BM*cg) x BN tile per K-slice unit
    const int64_t rows_per_tile = (int64_t)BM * p.cg;
    if (ok && a.ws)
        ok = encode_map(ctx, &L.tmW, TC_F32, a.ws, p.bn, (p.units - p.split_base) * rows_per_tile, p.bn, false, 1,
                        0, 32, 32, CU_TENSOR_MAP_SWIZZLE_128B);
    if (!ok) return TC_ERR_CUDA;
    if ((e = launch_mma(L, s->st)) != cudaSuccess) return TC_ERR_CUDA;
    ++launches;
    if (a.ws) {
        ReduceArgs r{};
        r.ws = a.ws;
        r.rows_per_tile = (int)rows_per_tile;
        r.bn = p.bn;
        r.first_tile = (int)(p.seg0_split > 1 ? 0 : p.seg0_tiles);
        r.ntiles = (int)(p.seg0_split > 1 ? p.seg0_tiles : p.tiles - p.seg0_tiles);
        r.S = p.seg0_split > 1 ? p.seg0_split : p.seg1_split;
        r.tiles_m = a.tiles_m;
        r.tiles_n = a.tiles_n;
        r.tiles_per_batch = a.tiles_per_batch;
        r.group_m = a.group_m;
        r.M = d->M;
        r.N = d->N;
        r.alpha = d->alpha;
        r.beta = d->beta;
        r.C = C;
        r.ldc = n.ldc;
        r.stride_c = a.stride_c;
        r.c_dtype = d->c_dtype;
        r.c_vec_ok = a.c_vec_ok;   // 16-byte vectors of 8 elements (two for fp32)
        r.bias = a.bias;
        r.act = a.act;
        r.col_scale = col_scale;
        r.int_sum = int_slices ? 1 : 0;
        // (r.status stays null: the stream's status word is mapped host
        // memory, and tc_stream_sync reports an expired wait, after which C
        // is undefined)
        if ((e = launch_reduce(r, s->st)) != cudaSuccess) return TC_ERR_CUDA;
        ++launches;
    }
    ctx->launches += launches;
    ctx->last = p.name;
    if (a.bias) ctx->last += "_bias";
    if (a.act == TC_ACT_GELU_TANH) ctx->last += "_gelu";
    return TC_OK;
}

// ----------------------------------------------------------- grouped launch

// One f16/bf16 problem of a grouped call, after validation.
struct GItem {
    int idx;                    // position in the caller's arrays
    Norm n;
    bool pack_a, pack_b;
    int64_t lda_p, ldb_p;       // leading dims of the operands the kernel reads
    size_t a_off, b_off;        // workspace offsets of the packed copies
    int64_t num_kb;
};

// Every f16/bf16 problem of a group goes through one batched repack launch
// (operands TMA cannot read in place) and one persistent tensor-core launch
// per GROUP_MAX problems, whose CTAs walk the tiles of all problems (tessl
// architecture.md, "Edge-Slice Support": ragged problems; one launch
// instead of one per problem removes the per-problem launch, pipeline fill
// and partial last wave).  Problems are ordered by K-loop length, longest
// first, so that the last waves hold the shortest tiles.
tc_status_t enqueue_grouped(tc_ctx *ctx, int n, const tc_gemm_desc *d, const void *const *A, const void *const *B,
                            void *const *C, const std::vector<int> &tc_idx, const std::vector<Norm> &norms,
                            tc_stream *s)
{
    const Force f = read_force();
    const int num_sms = f.sms > 0 ? f.sms : ctx->num_sms;
    std::vector<GItem> items;
    items.reserve(tc_idx.size());
    size_t ws_bytes = 0;
    for (int i : tc_idx) {
        GItem g{};
        g.idx = i;
        g.n = norms[i];
        g.pack_a = !aligned16(A[i]) || (g.n.lda % 8) != 0 || f.pack;
        g.pack_b = !aligned16(B[i]) || (g.n.ldb % 8) != 0 || f.pack;
        g.lda_p = g.pack_a ? (int64_t)round_up((size_t)g.n.a_cols, 64) : g.n.lda;
        g.ldb_p = g.pack_b ? (int64_t)round_up((size_t)g.n.b_cols, 64) : g.n.ldb;
        g.a_off = ws_bytes;
        if (g.pack_a) ws_bytes += round_up((size_t)(g.n.a_rows * g.lda_p * 2), 256);
        g.b_off = ws_bytes;
        if (g.pack_b) ws_bytes += round_up((size_t)(g.n.b_rows * g.ldb_p * 2), 256);
        g.num_kb = cdiv(d[i].K, BK);
        items.push_back(g);
    }
    (void)n;

    // kernel shape: the least modelled time over all problems' tiles
    static const int shapes[][2] = {{2, 256}, {1, 256}, {2, 128}, {1, 128}};
    int bn = 0, cg = 1;
    double best = 1e300;
    for (const auto &sh : shapes) {
        const int c = sh[0], b = sh[1];
        if (f.cg && c != f.cg) continue;
        if (f.bn && b != f.bn) continue;
        const int workers = c == 2 ? std::max(num_sms / 2, 1) : num_sms;
        double work = 0.0;
        int64_t tiles = 0;
        for (const GItem &g : items) {
            const int64_t t = cdiv(d[g.idx].M, BM * c) * cdiv(d[g.idx].N, b);
            tiles += t;
            work += (double)t * (double)g.num_kb;
        }
        const double waves = std::ceil((double)tiles / workers);
        const double t = std::max(work / workers, waves) * b / tile_rate(c, b);
        if (t < best - 1e-9) {
            best = t;
            bn = b;
            cg = c;
        }
    }
    if (bn == 0) return TC_ERR_VARIANT;

    tc_status_t st = ensure_ws(s, ws_bytes + 256);
    if (st != TC_OK) return st;
    uint8_t *ws = static_cast<uint8_t *>(s->ws);
    uint64_t launches = 0;
    cudaError_t e;

    // repack, PACK_MAX operands per launch
    {
        PackBatch pb;
        pb.count = 0;
        auto flush = [&]() -> bool {
            if (pb.count == 0) return true;
            if (launch_pack(pb, s->st) != cudaSuccess) return false;
            ++launches;
            pb.count = 0;
            return true;
        };
        for (const GItem &g : items) {
            if (g.pack_a) {
                pb.seg[pb.count++] = PackArgs{static_cast<const uint16_t *>(A[g.idx]),
                                              reinterpret_cast<uint16_t *>(ws + g.a_off), g.n.a_rows, g.n.a_cols,
                                              g.n.lda, g.lda_p, 0, 0, 1};
                if (pb.count == PACK_MAX && !flush()) return TC_ERR_CUDA;
            }
            if (g.pack_b) {
                pb.seg[pb.count++] = PackArgs{static_cast<const uint16_t *>(B[g.idx]),
                                              reinterpret_cast<uint16_t *>(ws + g.b_off), g.n.b_rows, g.n.b_cols,
                                              g.n.ldb, g.ldb_p, 0, 0, 1};
                if (pb.count == PACK_MAX && !flush()) return TC_ERR_CUDA;
            }
        }
        if (!flush()) return TC_ERR_CUDA;
    }

    std::stable_sort(items.begin(), items.end(),
                     [](const GItem &x, const GItem &y) { return x.num_kb > y.num_kb; });

    int pairs = 0;
    if (cg == 2) {
        int &mp = ctx->max_pairs[bn == 256 ? 2 : bn == 192 ? 1 : 0];
        if (mp < 0) mp = max_active_pairs(bn);
        if (mp < 1) return TC_ERR_VARIANT;
        pairs = mp;
    }
    const int workers = cg == 2 ? std::max(num_sms / 2, 1) : num_sms;
    std::unique_ptr<GroupTable> table(new GroupTable());
    for (size_t first = 0; first < items.size(); first += GROUP_MAX) {
        const size_t cnt = std::min(items.size() - first, (size_t)GROUP_MAX);
        GroupTable &gt = *table;
        std::memset(static_cast<void *>(&gt), 0, sizeof(GroupTable));
        gt.count = (int)cnt;
        int64_t units = 0, max_kb = 1;
        for (size_t j = 0; j < cnt; ++j) {
            const GItem &g = items[first + j];
            const tc_gemm_desc &q = d[g.idx];
            GroupInfo &gi = gt.info[j];
            gi.M = q.M;
            gi.N = q.N;
            gi.num_kb = (int)g.num_kb;
            gi.tiles_m = (int)cdiv(q.M, BM * cg);
            gi.tiles_n = (int)cdiv(q.N, bn);
            gi.unit_begin = (int)units;
            units += (int64_t)gi.tiles_m * gi.tiles_n;
            if (units > INT32_MAX / 2) return TC_ERR_OVERFLOW;
            max_kb = std::max<int64_t>(max_kb, g.num_kb);
            gi.a_kmajor = !q.transpose_a;
            gi.b_kmajor = q.transpose_b;
            const uint32_t fmt = q.a_dtype == TC_BF16 ? 1u : 0u;
            gi.idesc = (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(!gi.a_kmajor) << 15) |
                       ((uint32_t)(!gi.b_kmajor) << 16) | ((uint32_t)(bn >> 3) << 17) |
                       ((uint32_t)((BM * cg) >> 4) << 24);
            gi.c_dtype = q.c_dtype;
            const int64_t ec = (int64_t)elem_size(q.c_dtype);
            gi.c_vec_ok = aligned16(C[g.idx]) && (g.n.ldc * ec) % 16 == 0;
            gi.c_tma = gi.c_vec_ok && !f.direct_store;
            gi.alpha = q.alpha;
            gi.beta = q.beta;
            gi.C = C[g.idx];
            gi.ldc = g.n.ldc;
            const void *Au = g.pack_a ? static_cast<const void *>(ws + g.a_off) : A[g.idx];
            const void *Bu = g.pack_b ? static_cast<const void *>(ws + g.b_off) : B[g.idx];
            bool ok = gi.a_kmajor
                          ? encode_map(ctx, &gt.tmA[j], q.a_dtype, Au, q.K, q.M, g.lda_p, false, 1, 0, 64, BM)
                          : encode_map(ctx, &gt.tmA[j], q.a_dtype, Au, q.M, q.K, g.lda_p, false, 1, 0, 64, 64);
            if (ok)
                ok = gi.b_kmajor ? encode_map(ctx, &gt.tmB[j], q.a_dtype, Bu, q.K, q.N, g.ldb_p, false, 1, 0, 64,
                                              (uint32_t)(bn / cg))
                                 : encode_map(ctx, &gt.tmB[j], q.a_dtype, Bu, q.N, q.K, g.ldb_p, false, 1, 0, 64, 64);
            if (ok && gi.c_tma)
                ok = encode_map(ctx, &gt.tmC[j], q.c_dtype, C[g.idx], q.N, q.M, g.n.ldc, false, 1, 0, 32, 32,
                                q.c_dtype == TC_F32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
            if (!ok) return TC_ERR_CUDA;
        }
        MmaLaunch L{};
        L.bn = bn;
        L.cg = cg;
        int grid = (int)std::min<int64_t>(units, workers);
        if (f.grid > 0) grid = (int)std::min<int64_t>(f.grid, units);
        if (cg == 2) grid = std::min(grid, pairs);
        L.grid = grid * cg;
        MmaArgs &a = L.args;
        a.num_kb = (int)max_kb;
        a.batch = 1;
        a.seg0_tiles = (int)units;
        a.seg0_split = 1;
        a.seg1_split = 1;
        a.split_base = (int)units;
        a.total_units = (int)units;
        a.group_m = f.group_m > 0 ? f.group_m : 4;
        a.status = s->status_dev;
        a.timeout_ns = 4000000000ull + (unsigned long long)max_kb * 20000ull;
        if (f.debug_timeout_ms > 0) a.timeout_ns = (unsigned long long)f.debug_timeout_ms * 1000000ull;
        a.debug_drop_tfull = f.debug_drop;
        if ((e = launch_mma_grouped(L, gt, s->st)) != cudaSuccess) return TC_ERR_CUDA;
        ++launches;
    }
    char buf[96];
    std::snprintf(buf, sizeof buf, "grouped_tcgen05_%dx%d%s_n%d", BM * cg, bn, cg == 2 ? "_pair" : "",
                  (int)items.size());
    ctx->launches += launches;
    ctx->last = buf;
    return TC_OK;
}

// The fused epilogue's own checks (after the GEMM's): an activation this
// library knows, a tensor-core path to fuse into, a bias apart from C.
tc_status_t validate_epilogue(const tc_gemm_desc *d, const Norm &n, const tc_epilogue *epi, const void *C)
{
    if (!epi) return TC_ERR_NULL;
    if (epi->activation != TC_ACT_NONE && epi->activation != TC_ACT_GELU_TANH) return TC_ERR_EPILOGUE;
    if (d->a_dtype == TC_F32) return TC_ERR_EPILOGUE;
    if (epi->bias && ranges_overlap(epi->bias, (int64_t)d->N * (int64_t)elem_size(d->c_dtype), C, n.c_bytes))
        return TC_ERR_OVERLAP;
    return TC_OK;
}

tc_status_t run(tc_ctx *ctx, const tc_gemm_desc *d, const void *A, const void *B, void *C, int64_t batch,
                int64_t sa, int64_t sb, int64_t sc, tc_stream *s, const tc_epilogue *epi = nullptr)
{
    if (!ctx || !s) return TC_ERR_NULL;
    Norm n;
    tc_status_t st = validate(d, A, B, C, batch, sa, sb, sc, &n);
    if (st != TC_OK) return st;
    if (epi && (st = validate_epilogue(d, n, epi, C)) != TC_OK) return st;
    Plan p;
    if ((st = make_plan(d, n, A, B, ctx->num_sms, &p, epi == nullptr)) != TC_OK) return st;
    std::lock_guard<std::mutex> g(ctx->mu);
    if (cudaSetDevice(ctx->device) != cudaSuccess) return TC_ERR_CUDA;
    return enqueue(ctx, d, n, p, A, B, C, s, epi);
}

// ------------------------------------------------------------ relaxed fp32
// tessl architecture.md, "GEMM Pipeline & Kernel Selection": a relaxed
// precision mode beside f32-exact for fp32 operands.  Here each fp32 value
// x = hi + lo + e (hi = bf16(x), lo = bf16(x - hi), |e| <= 2^-16 |x|), and
// op(A) op(B) ~= A_hi B_hi + A_hi B_lo + A_lo B_hi is ONE bf16 tensor-core
// GEMM over K' = 3K of [A_hi | A_hi | A_lo] and [B_hi ; B_lo ; B_hi]: every
// product is exact in fp32, the dropped terms are below 2^-15 |a b|, so the
// result meets the 1e-4 * sum|ab| bound of the non-exact paths.

tc_status_t ensure_rx(tc_stream *s, size_t bytes)
{
    if (bytes <= s->rx_cap) return TC_OK;
    const size_t cap = round_up(bytes + bytes / 4, (size_t)1 << 20);
    if (s->rx) {
        cudaError_t e = cudaFreeAsync(s->rx, s->st);
        s->rx = nullptr;
        s->rx_cap = 0;
        if (e != cudaSuccess) return TC_ERR_CUDA;
    }
    if (cudaMallocAsync(&s->rx, cap, s->st) != cudaSuccess) {
        s->rx = nullptr;
        return TC_ERR_CUDA;
    }
    s->rx_cap = cap;
    return TC_OK;
}

tc_status_t run_relaxed(tc_ctx *ctx, const tc_gemm_desc *d, const tc_epilogue *epi, const void *A, const void *B,
                        void *C, tc_stream *s)
{
    if (!ctx || !s) return TC_ERR_NULL;
    Norm n;
    tc_status_t st = validate(d, A, B, C, 1, 0, 0, 0, &n);
    if (st != TC_OK) return st;
    if (d->a_dtype != TC_F32) return TC_ERR_DTYPE;
    if (epi) {
        if (epi->activation != TC_ACT_NONE && epi->activation != TC_ACT_GELU_TANH) return TC_ERR_EPILOGUE;
        if (epi->bias && ranges_overlap(epi->bias, (int64_t)d->N * 4, C, n.c_bytes)) return TC_ERR_OVERLAP;
    }
    if ((int64_t)d->K * 3 > INT32_MAX) return TC_ERR_OVERFLOW;
    // the split copies: the K dimension (A's columns unless transposed, B's
    // rows unless transposed) tripled, rows padded to 64 elements
    const bool a_kcols = !d->transpose_a, b_kcols = d->transpose_b;
    const int64_t a_rows = a_kcols ? n.a_rows : 3 * n.a_rows, a_cols = a_kcols ? 3 * n.a_cols : n.a_cols;
    const int64_t b_rows = b_kcols ? n.b_rows : 3 * n.b_rows, b_cols = b_kcols ? 3 * n.b_cols : n.b_cols;
    const int64_t lda2 = (int64_t)round_up((size_t)a_cols, 64), ldb2 = (int64_t)round_up((size_t)b_cols, 64);
    if (lda2 > INT32_MAX || ldb2 > INT32_MAX) return TC_ERR_OVERFLOW;
    const size_t a_bytes = round_up((size_t)(a_rows * lda2 * 2), 256), b_bytes = (size_t)(b_rows * ldb2 * 2);

    tc_gemm_desc d2 = *d;
    d2.a_dtype = d2.b_dtype = TC_BF16;
    d2.K = 3 * d->K;
    d2.lda = (int32_t)lda2;
    d2.ldb = (int32_t)ldb2;
    d2.ldc = (int32_t)n.ldc;
    tc_epilogue e2{};
    if (epi) e2 = *epi;

    std::lock_guard<std::mutex> g(ctx->mu);
    if (cudaSetDevice(ctx->device) != cudaSuccess) return TC_ERR_CUDA;
    if ((st = ensure_rx(s, a_bytes + b_bytes)) != TC_OK) return st;
    uint16_t *A2 = static_cast<uint16_t *>(s->rx);
    uint16_t *B2 = reinterpret_cast<uint16_t *>(static_cast<uint8_t *>(s->rx) + a_bytes);
    Norm n2;
    if ((st = validate(&d2, A2, B2, C, 1, 0, 0, 0, &n2)) != TC_OK) return st;
    Plan p2;
    if ((st = make_plan(&d2, n2, A2, B2, ctx->num_sms, &p2, false)) != TC_OK) return st;
    const SplitArgs sa{static_cast<const float *>(A), A2, n.a_rows, n.a_cols, n.lda, lda2, a_kcols ? 1 : 0, {0, 0, 1}};
    const SplitArgs sb{static_cast<const float *>(B), B2, n.b_rows, n.b_cols, n.ldb, ldb2, b_kcols ? 1 : 0, {0, 1, 0}};
    if (launch_split(sa, s->st) != cudaSuccess || launch_split(sb, s->st) != cudaSuccess) return TC_ERR_CUDA;
    ctx->launches += 2;
    st = enqueue(ctx, &d2, n2, p2, A2, B2, C, s, epi ? &e2 : nullptr);
    if (st == TC_OK) ctx->last = "relaxed_f32_3xbf16_" + ctx->last;
    return st;
}

// ---------------------------------------------------------------- int8 GEMM
// tessl architecture.md, "Integer GEMM": int8 x int8 summed exactly, then
// per-column dequantisation.  Both operands are widened to bf16 (exact for
// int8) and run through the bf16 tensor-core kernel with K cut into slices
// of at most 16 K blocks (1024 products, |sum| <= 2^24: exact in the fp32
// accumulator); the reduction kernel adds the slices as 64-bit integers,
// rounds once to fp32, scales by the column's factor, then alpha/beta.

tc_status_t run_i8(tc_ctx *ctx, const tc_gemm_desc *d, const float *col_scale, const void *A, const void *B,
                   void *C, tc_stream *s)
{
    if (!ctx || !s) return TC_ERR_NULL;
    Norm n;
    tc_status_t st = validate(d, A, B, C, 1, 0, 0, 0, &n, V_I8);
    if (st != TC_OK) return st;
    if (d->a_dtype != TC_I8) return TC_ERR_DTYPE;
    if (!col_scale) return TC_ERR_NULL;
    if (d->K > I8_K_MAX) return TC_ERR_DIM;
    if (ranges_overlap(col_scale, (int64_t)d->N * 4, C, n.c_bytes)) return TC_ERR_OVERLAP;
    const int64_t lda2 = (int64_t)round_up((size_t)n.a_cols, 64), ldb2 = (int64_t)round_up((size_t)n.b_cols, 64);
    const size_t a_bytes = round_up((size_t)(n.a_rows * lda2 * 2), 256), b_bytes = (size_t)(n.b_rows * ldb2 * 2);
    tc_gemm_desc d2 = *d;
    d2.a_dtype = d2.b_dtype = TC_BF16;
    d2.accum_dtype = TC_F32;
    d2.lda = (int32_t)lda2;
    d2.ldb = (int32_t)ldb2;
    d2.ldc = (int32_t)n.ldc;

    std::lock_guard<std::mutex> g(ctx->mu);
    if (cudaSetDevice(ctx->device) != cudaSuccess) return TC_ERR_CUDA;
    if ((st = ensure_rx(s, a_bytes + b_bytes)) != TC_OK) return st;
    uint16_t *A2 = static_cast<uint16_t *>(s->rx);
    uint16_t *B2 = reinterpret_cast<uint16_t *>(static_cast<uint8_t *>(s->rx) + a_bytes);
    Norm n2;
    if ((st = validate(&d2, A2, B2, C, 1, 0, 0, 0, &n2)) != TC_OK) return st;
    Plan p;
    if ((st = make_plan(&d2, n2, A2, B2, ctx->num_sms, &p, false)) != TC_OK) return st;
    p.csplit = false;      // integer slices are added through memory (or on chip in TMEM)
    const int64_t num_kb = cdiv(d->K, BK);
    const int S = (int)cdiv(num_kb, I8_SLICE_KB);
    char buf[48];
    const Force f = read_force();
    if (d->K <= I8_ONCHIP_K_MAX && f.i8acc != 0) {
        // one unit per tile, its K slices summed as int32 in TMEM (|sum| <=
        // 2^14 K <= 2^30): 128-wide tiles (two accumulators and the sums
        // fit in TMEM), CTA pairs unless that leaves half the SMs idle
        const int64_t tiles2 = cdiv(d->M, 2 * BM) * cdiv(d->N, 128);
        p.cg = (tiles2 * 2 >= ctx->num_sms) ? 2 : 1;
        p.bn = 128;
        p.i8acc = true;
        const int64_t tiles = cdiv(d->M, BM * p.cg) * cdiv(d->N, 128);
        p.tiles = p.seg0_tiles = tiles;
        p.seg0_split = p.seg1_split = 1;
        p.split_base = tiles;
        p.units = tiles;
        p.split = 1;
        std::snprintf(buf, sizeof buf, "_i8acc_s%d", S);
        p.name = std::string("tcgen05_") + (d->transpose_a ? (d->transpose_b ? "tt" : "tn") : (d->transpose_b ? "nt" : "nn")) +
                 "_bf16_" + (d->c_dtype == TC_F32 ? "f32" : d->c_dtype == TC_BF16 ? "bf16" : "f16") +
                 (p.cg == 2 ? "_256x128_pair" : "_128x128");
    } else {
        // every tile in the same K slices of at most I8_SLICE_KB blocks (the
        // plan's own tail split would add its slices in fp32)
        const int64_t tiles = cdiv(d->M, BM * p.cg) * cdiv(d->N, p.bn);
        p.tiles = tiles;
        p.seg0_tiles = tiles;
        p.seg0_split = S;
        p.seg1_split = 1;
        p.split_base = 0;
        p.units = tiles * S;
        p.split = S > 1 ? 2 : 1;
        std::snprintf(buf, sizeof buf, "_i8s%d", S);
    }
    if (p.units > INT32_MAX / 2) return TC_ERR_OVERFLOW;
    const int workers = p.cg == 2 ? std::max(ctx->num_sms / 2, 1) : ctx->num_sms;
    p.grid = (int)std::min<int64_t>(p.units, workers) * p.cg;
    const WidenArgs wa{static_cast<const int8_t *>(A), A2, n.a_rows, n.a_cols, n.lda, lda2, 0};
    const WidenArgs wb{static_cast<const int8_t *>(B), B2, n.b_rows, n.b_cols, n.ldb, ldb2, 0};
    if (launch_widen(wa, s->st) != cudaSuccess || launch_widen(wb, s->st) != cudaSuccess) return TC_ERR_CUDA;
    ctx->launches += 2;
    st = enqueue(ctx, &d2, n2, p, A2, B2, C, s, nullptr, col_scale, true);
    if (st == TC_OK) ctx->last = "i8_dequant_" + ctx->last.substr(0, ctx->last.find("_tail")) + buf;
    return st;
}

// ---------------------------------------------------- int8-weight product
// Foundry metal.md, "Custom Compute Kernels" (fm_sgemm_q8, fm_matvec_q8):
// Out = X @ (W_q8 * scale[n])^T; tensorcore gemm.md "Kernel variants": the
// M <= 4 GEMV over Q8 weights.  Up to GEMV_MAX_ROWS activation rows the
// skinny-product kernel streams the int8 weights once and widens them in
// registers; beyond, the weights are widened once (exactly) to the
// activations' type and the tensor-core GEMM applies the scales in its
// epilogue.

tc_status_t run_q8w(tc_ctx *ctx, const tc_gemm_desc *d, const float *scale, const void *X, const void *W, void *C,
                    tc_stream *s)
{
    if (!ctx || !s) return TC_ERR_NULL;
    Norm n;
    tc_status_t st = validate(d, X, W, C, 1, 0, 0, 0, &n, V_Q8W);
    if (st != TC_OK) return st;
    if (!scale) return TC_ERR_NULL;
    if (ranges_overlap(scale, (int64_t)d->N * 4, C, n.c_bytes)) return TC_ERR_OVERLAP;
    const Force f = read_force();
    const char *dt = d->a_dtype == TC_BF16 ? "bf16" : "f16";
    const char *ct = d->c_dtype == TC_F32 ? "f32" : dt;
    char buf[96];
    if (d->M <= GEMV_MAX_ROWS && f.gemv != 0) {
        GemvArgs g{};
        g.X = X;
        g.W = W;
        g.C = C;
        g.scale = scale;
        g.rows_x = d->M;
        g.rows_w = d->N;
        g.K = d->K;
        g.ldx = n.lda;
        g.ldw = n.ldb;
        g.c_sx = n.ldc;
        g.c_sw = 1;
        g.c_dtype = d->c_dtype;
        g.alpha = d->alpha;
        g.beta = d->beta;
        g.x_vec = aligned16(X) && (n.lda * 2) % 16 == 0;
        g.w_vec = aligned16(W) && n.ldb % 16 == 0;
        g.w_i8 = 1;
        g.x_bf16 = d->a_dtype == TC_BF16;
        g.ksplit = f.gemv_ks > 0 ? pow2_floor(std::min(f.gemv_ks, 8)) : gemv_ksplit(d->N, d->K, true, ctx->num_sms);
        std::snprintf(buf, sizeof buf, "gemv_q8w_nt_%s_%s_x%d", dt, ct, (int)d->M);
        std::string name = buf;
        std::lock_guard<std::mutex> lk(ctx->mu);
        if (cudaSetDevice(ctx->device) != cudaSuccess) return TC_ERR_CUDA;
        if ((st = enqueue_gemv(ctx, s, g, f, name)) != TC_OK) return st;
        ctx->last = name;
        return TC_OK;
    }
    // W [N, K] int8 -> the activations' type, rows padded to 64 elements
    const int64_t ldb2 = (int64_t)round_up((size_t)d->K, 64);
    if (ldb2 > INT32_MAX) return TC_ERR_OVERFLOW;
    const size_t w_bytes = (size_t)(d->N * ldb2 * 2);
    tc_gemm_desc d2 = *d;
    d2.b_dtype = d->a_dtype;
    d2.ldb = (int32_t)ldb2;
    d2.lda = (int32_t)n.lda;
    d2.ldc = (int32_t)n.ldc;
    std::lock_guard<std::mutex> lk(ctx->mu);
    if (cudaSetDevice(ctx->device) != cudaSuccess) return TC_ERR_CUDA;
    if ((st = ensure_rx(s, w_bytes)) != TC_OK) return st;
    uint16_t *W2 = static_cast<uint16_t *>(s->rx);
    Norm n2;
    if ((st = validate(&d2, X, W2, C, 1, 0, 0, 0, &n2)) != TC_OK) return st;
    Plan p;
    if ((st = make_plan(&d2, n2, X, W2, ctx->num_sms, &p, false)) != TC_OK) return st;
    const WidenArgs wa{static_cast<const int8_t *>(W), W2, d->N, d->K, n.ldb, ldb2, d->a_dtype == TC_F16 ? 1 : 0};
    if (launch_widen(wa, s->st) != cudaSuccess) return TC_ERR_CUDA;
    ctx->launches += 1;
    st = enqueue(ctx, &d2, n2, p, X, W2, C, s, nullptr, scale, false);
    if (st == TC_OK) ctx->last = "q8w_widen_" + ctx->last;
    return st;
}

tc_status_t stream_init(tc_ctx *ctx, tc_stream *s)
{
    s->ctx = ctx;
    if (cudaHostAlloc(reinterpret_cast<void **>(&s->status_host), sizeof(unsigned), cudaHostAllocMapped) !=
        cudaSuccess)
        return TC_ERR_CUDA;
    *s->status_host = 0u;
    if (cudaHostGetDevicePointer(reinterpret_cast<void **>(&s->status_dev), s->status_host, 0) != cudaSuccess)
        return TC_ERR_CUDA;
    return TC_OK;
}

void stream_free(tc_stream *s)
{
    if (!s) return;
    if (s->st) cudaStreamSynchronize(s->st);
    if (s->ws) cudaFree(s->ws);
    if (s->rx) cudaFree(s->rx);
    if (s->status_host) cudaFreeHost(s->status_host);
    if (s->owned && s->st) cudaStreamDestroy(s->st);
    delete s;
}

}  // namespace

// =============================================================== C ABI

extern "C" {

const char *tc_status_string(tc_status_t st)
{
    switch (st) {
    case TC_OK: return "ok";
    case TC_ERR_NULL: return "null pointer";
    case TC_ERR_DIM: return "dimension out of range (M, N, K, batch must be >= 1)";
    case TC_ERR_LD: return "leading dimension below its minimum or negative";
    case TC_ERR_DTYPE: return "unsupported dtype combination";
    case TC_ERR_SCALAR: return "alpha or beta is not finite";
    case TC_ERR_OVERLAP: return "C overlaps A or B";
    case TC_ERR_OVERFLOW: return "size computation overflows";
    case TC_ERR_ALIGN_UNSUPPORTED: return "alignment unsupported";
    case TC_ERR_CUDA: return "CUDA error";
    case TC_ERR_DEVICE_TIMEOUT: return "device wait timed out; the kernel stopped early";
    case TC_ERR_STRIDE: return "invalid batch stride";
    case TC_ERR_VARIANT: return "forced variant cannot serve this problem";
    case TC_ERR_SCRATCH: return "problem needs more scratch than the static buffer of tc_gemm_splitk_noalloc holds";
    case TC_ERR_EPILOGUE: return "fused epilogue refused: unknown activation, or f32 operands (exact-fp32 path)";
    case TC_ERR_LAYOUT: return "transpose flags this call does not support";
    }
    return "unknown status";
}

tc_status_t tc_ctx_create(tc_ctx **out, int device)
{
    if (!out) return TC_ERR_NULL;
    *out = nullptr;
    int count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess || device < 0 || device >= count) {
        cudaGetLastError();
        return TC_ERR_CUDA;
    }
    if (cudaSetDevice(device) != cudaSuccess) return TC_ERR_CUDA;
    tc_ctx *ctx = new tc_ctx();
    ctx->device = device;
    if (cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
        delete ctx;
        return TC_ERR_CUDA;
    }
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn) {
        delete ctx;
        return TC_ERR_CUDA;
    }
    ctx->encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    tc_stream *s = new tc_stream();
    tc_status_t st = stream_init(ctx, s);
    if (st == TC_OK && cudaStreamCreateWithFlags(&s->st, cudaStreamNonBlocking) != cudaSuccess) st = TC_ERR_CUDA;
    if (st != TC_OK) {
        stream_free(s);
        delete ctx;
        return st;
    }
    s->owned = true;
    ctx->def = s;
    *out = ctx;
    return TC_OK;
}

void tc_ctx_destroy(tc_ctx *ctx)
{
    if (!ctx) return;
    cudaSetDevice(ctx->device);
    stream_free(ctx->def);
    for (int i = 0; i < 3; ++i)
        if (ctx->dbuf[i]) cudaFree(ctx->dbuf[i]);
    if (ctx->copy_in) cudaStreamDestroy(ctx->copy_in);
    if (ctx->copy_out) cudaStreamDestroy(ctx->copy_out);
    for (cudaEvent_t e : ctx->host_ev) cudaEventDestroy(e);
    delete ctx;
}

tc_status_t tc_stream_create(tc_ctx *ctx, tc_stream **out)
{
    if (!ctx || !out) return TC_ERR_NULL;
    *out = nullptr;
    if (cudaSetDevice(ctx->device) != cudaSuccess) return TC_ERR_CUDA;
    tc_stream *s = new tc_stream();
    tc_status_t st = stream_init(ctx, s);
    if (st == TC_OK && cudaStreamCreateWithFlags(&s->st, cudaStreamNonBlocking) != cudaSuccess) st = TC_ERR_CUDA;
    if (st != TC_OK) {
        stream_free(s);
        return st;
    }
    s->owned = true;
    *out = s;
    return TC_OK;
}

tc_status_t tc_stream_wrap(tc_ctx *ctx, void *cuda_stream, tc_stream **out)
{
    if (!ctx || !out) return TC_ERR_NULL;
    *out = nullptr;
    if (cudaSetDevice(ctx->device) != cudaSuccess) return TC_ERR_CUDA;
    tc_stream *s = new tc_stream();
    tc_status_t st = stream_init(ctx, s);
    if (st != TC_OK) {
        stream_free(s);
        return st;
    }
    s->st = static_cast<cudaStream_t>(cuda_stream);
    s->owned = false;
    *out = s;
    return TC_OK;
}

tc_status_t tc_stream_sync(tc_stream *s)
{
    if (!s) return TC_ERR_NULL;
    if (cudaStreamSynchronize(s->st) != cudaSuccess) return TC_ERR_CUDA;
    return read_status(s);
}

void *tc_stream_handle(tc_stream *s) { return s ? static_cast<void *>(s->st) : nullptr; }

void tc_stream_destroy(tc_stream *s) { stream_free(s); }

tc_status_t tc_gemm_async(tc_ctx *ctx, const tc_gemm_desc *d, const void *A, const void *B, void *C,
                          tc_stream *s)
{
    return run(ctx, d, A, B, C, 1, 0, 0, 0, s);
}

tc_status_t tc_gemm(tc_ctx *ctx, const tc_gemm_desc *d, const void *A, const void *B, void *C)
{
    if (!ctx) return TC_ERR_NULL;
    tc_status_t st = run(ctx, d, A, B, C, 1, 0, 0, 0, ctx->def);
    if (st != TC_OK) return st;
    return tc_stream_sync(ctx->def);
}

tc_status_t tc_gemm_epilogue_async(tc_ctx *ctx, const tc_gemm_desc *d, const tc_epilogue *epi, const void *A,
                                   const void *B, void *C, tc_stream *s)
{
    if (!epi) return TC_ERR_NULL;
    return run(ctx, d, A, B, C, 1, 0, 0, 0, s, epi);
}

tc_status_t tc_gemm_epilogue(tc_ctx *ctx, const tc_gemm_desc *d, const tc_epilogue *epi, const void *A,
                             const void *B, void *C)
{
    if (!ctx) return TC_ERR_NULL;
    tc_status_t st = tc_gemm_epilogue_async(ctx, d, epi, A, B, C, ctx->def);
    if (st != TC_OK) return st;
    return tc_stream_sync(ctx->def);
}

tc_status_t tc_gemm_f32_relaxed_async(tc_ctx *ctx, const tc_gemm_desc *d, const tc_epilogue *epi, const void *A,
                                      const void *B, void *C, tc_stream *s)
{
    return run_relaxed(ctx, d, epi, A, B, C, s);
}

tc_status_t tc_gemm_f32_relaxed(tc_ctx *ctx, const tc_gemm_desc *d, const tc_epilogue *epi, const void *A,
                                const void *B, void *C)
{
    if (!ctx) return TC_ERR_NULL;
    tc_status_t st = run_relaxed(ctx, d, epi, A, B, C, ctx->def);
    if (st != TC_OK) return st;
    return tc_stream_sync(ctx->def);
}

tc_status_t tc_gemm_i8_dequant_async(tc_ctx *ctx, const tc_gemm_desc *d, const float *col_scale, const void *A,
                                     const void *B, void *C, tc_stream *s)
{
    return run_i8(ctx, d, col_scale, A, B, C, s);
}

tc_status_t tc_gemm_i8_dequant(tc_ctx *ctx, const tc_gemm_desc *d, const float *col_scale, const void *A,
                               const void *B, void *C)
{
    if (!ctx) return TC_ERR_NULL;
    tc_status_t st = run_i8(ctx, d, col_scale, A, B, C, ctx->def);
    if (st != TC_OK) return st;
    return tc_stream_sync(ctx->def);
}

tc_status_t tc_gemm_q8_weight_async(tc_ctx *ctx, const tc_gemm_desc *d, const float *scale, const void *X,
                                    const void *W, void *C, tc_stream *s)
{
    return run_q8w(ctx, d, scale, X, W, C, s);
}

tc_status_t tc_gemm_q8_weight(tc_ctx *ctx, const tc_gemm_desc *d, const float *scale, const void *X, const void *W,
                              void *C)
{
    if (!ctx) return TC_ERR_NULL;
    tc_status_t st = run_q8w(ctx, d, scale, X, W, C, ctx->def);
    if (st != TC_OK) return st;
    return tc_stream_sync(ctx->def);
}

tc_status_t tc_gemm_q8_weight_validate(const tc_gemm_desc *d, const float *scale, const void *X, const void *W,
                                       const void *C)
{
    Norm n;
    tc_status_t st = validate(d, X, W, C, 1, 0, 0, 0, &n, V_Q8W);
    if (st != TC_OK) return st;
    if (!scale) return TC_ERR_NULL;
    if (ranges_overlap(scale, (int64_t)d->N * 4, C, n.c_bytes)) return TC_ERR_OVERLAP;
    return TC_OK;
}

tc_status_t tc_gemm_batched_async(tc_ctx *ctx, const tc_gemm_batched_desc *bd, const void *A, const void *B,
                                  void *C, tc_stream *s)
{
    if (!bd) return TC_ERR_NULL;
    return run(ctx, &bd->base, A, B, C, bd->batch, bd->stride_a, bd->stride_b, bd->stride_c, s);
}

tc_status_t tc_gemm_batched(tc_ctx *ctx, const tc_gemm_batched_desc *bd, const void *A, const void *B, void *C)
{
    if (!ctx) return TC_ERR_NULL;
    tc_status_t st = tc_gemm_batched_async(ctx, bd, A, B, C, ctx->def);
    if (st != TC_OK) return st;
    return tc_stream_sync(ctx->def);
}

tc_status_t tc_gemm_grouped_async(tc_ctx *ctx, int n, const tc_gemm_desc *d, const void *const *A,
                                  const void *const *B, void *const *C, tc_stream *s)
{
    if (!ctx || !s || !d || !A || !B || !C) return TC_ERR_NULL;
    if (n < 0) return TC_ERR_DIM;
    // validate everything before enqueueing anything
    std::vector<Norm> norms((size_t)n);
    std::vector<int> tc_idx, other_idx;
    for (int i = 0; i < n; ++i) {
        tc_status_t st = validate(&d[i], A[i], B[i], C[i], 1, 0, 0, 0, &norms[(size_t)i]);
        if (st != TC_OK) return st;
        (d[i].a_dtype == TC_F32 ? other_idx : tc_idx).push_back(i);
    }
    // a lone tensor-core problem takes the single-problem dispatcher
    if (tc_idx.size() < 2 || read_force().grouped == 0) {
        other_idx.insert(other_idx.end(), tc_idx.begin(), tc_idx.end());
        tc_idx.clear();
    }
    for (int i : other_idx) {
        tc_status_t st = run(ctx, &d[i], A[i], B[i], C[i], 1, 0, 0, 0, s);
        if (st != TC_OK) return st;
    }
    if (tc_idx.empty()) return TC_OK;
    std::lock_guard<std::mutex> g(ctx->mu);
    if (cudaSetDevice(ctx->device) != cudaSuccess) return TC_ERR_CUDA;
    return enqueue_grouped(ctx, n, d, A, B, C, tc_idx, norms, s);
}

tc_status_t tc_gemm_host(tc_ctx *ctx, const tc_gemm_desc *d, const void *A_host, const void *B_host, void *C_host)
{
    if (!ctx) return TC_ERR_NULL;
    std::lock_guard<std::mutex> host_lock(ctx->host_mu);
    Norm n;
    // validate on the host buffers (overlap between host ranges, dims, ...)
    tc_status_t st = validate(d, A_host, B_host, C_host, 1, 0, 0, 0, &n);
    if (st != TC_OK) return st;
    const size_t bytes[3] = {(size_t)n.a_bytes, (size_t)n.b_bytes, (size_t)n.c_bytes};
    {
        std::lock_guard<std::mutex> g(ctx->mu);
        if (cudaSetDevice(ctx->device) != cudaSuccess) return TC_ERR_CUDA;
        for (int i = 0; i < 3; ++i) {
            if (bytes[i] > ctx->dcap[i]) {
                if (ctx->dbuf[i]) cudaFree(ctx->dbuf[i]);
                ctx->dbuf[i] = nullptr;
                ctx->dcap[i] = 0;
                if (cudaMalloc(&ctx->dbuf[i], bytes[i]) != cudaSuccess) return TC_ERR_CUDA;
                ctx->dcap[i] = bytes[i];
            }
        }
        if ((!ctx->copy_in && cudaStreamCreateWithFlags(&ctx->copy_in, cudaStreamNonBlocking) != cudaSuccess) ||
            (!ctx->copy_out && cudaStreamCreateWithFlags(&ctx->copy_out, cudaStreamNonBlocking) != cudaSuccess))
            return TC_ERR_CUDA;
    }
    // The device copies keep the host layouts (same leading dimensions).  A
    // is moved in bands of op(A) rows and C in the same bands, so that the
    // GEMM of band i runs while band i + 1 arrives and band i - 1 returns:
    // B (needed whole) first, then band by band on the copy-in stream; each
    // band's GEMM on the context's stream once its band has landed; each
    // band of C back on the copy-out stream once its GEMM is done.
    // (Host-device copies run at one rate per direction whatever the number
    // of streams; the two directions overlap.)
    const int64_t es_a = (int64_t)elem_size(d->a_dtype), es_c = (int64_t)elem_size(d->c_dtype);
    const int64_t hb = read_force().host_band;
    const int64_t band = hb > 0 ? std::min<int64_t>(hb, d->M)
                         : d->M <= 1536 ? d->M : std::max<int64_t>(1024, (int64_t)round_up((size_t)cdiv(d->M, 4), 256));
    const int nb = (int)cdiv(d->M, band);
    uint8_t *dA = static_cast<uint8_t *>(ctx->dbuf[0]), *dB = static_cast<uint8_t *>(ctx->dbuf[1]);
    uint8_t *dC = static_cast<uint8_t *>(ctx->dbuf[2]);
    const uint8_t *hA = static_cast<const uint8_t *>(A_host);
    uint8_t *hC = static_cast<uint8_t *>(C_host);
    cudaStream_t comp = ctx->def->st;
    // events from the context's pool, created on first use and re-recorded
    // by later calls (each call has synchronised all three streams before it
    // returns, so no earlier record is still pending)
    size_t next_ev = 0;
    auto event = [&](cudaEvent_t *e) {
        if (next_ev == ctx->host_ev.size()) {
            cudaEvent_t fresh;
            if (cudaEventCreateWithFlags(&fresh, cudaEventDisableTiming) != cudaSuccess) return false;
            ctx->host_ev.push_back(fresh);
        }
        *e = ctx->host_ev[next_ev++];
        return true;
    };
    auto finish = [&](tc_status_t result) {
        cudaStreamSynchronize(ctx->copy_in);
        cudaStreamSynchronize(ctx->copy_out);
        tc_status_t s2 = tc_stream_sync(ctx->def);
        return result != TC_OK ? result : s2;
    };
    // one band of op(A) rows [m0, m1): rows of A, or columns of A stored [K, M]
    auto copy_a = [&](int64_t m0, int64_t m1) {
        if (!d->transpose_a)
            return cudaMemcpy2DAsync(dA + m0 * n.lda * es_a, n.lda * es_a, hA + m0 * n.lda * es_a, n.lda * es_a,
                                     n.a_cols * es_a, m1 - m0, cudaMemcpyHostToDevice, ctx->copy_in);
        return cudaMemcpy2DAsync(dA + m0 * es_a, n.lda * es_a, hA + m0 * es_a, n.lda * es_a, (m1 - m0) * es_a,
                                 n.a_rows, cudaMemcpyHostToDevice, ctx->copy_in);
    };
    auto copy_c = [&](int64_t m0, int64_t m1, cudaMemcpyKind kind, cudaStream_t str) {
        uint8_t *dst = kind == cudaMemcpyHostToDevice ? dC + m0 * n.ldc * es_c : hC + m0 * n.ldc * es_c;
        const uint8_t *src = kind == cudaMemcpyHostToDevice ? hC + m0 * n.ldc * es_c : dC + m0 * n.ldc * es_c;
        return cudaMemcpy2DAsync(dst, n.ldc * es_c, src, n.ldc * es_c, d->N * es_c, m1 - m0, kind, str);
    };
    cudaEvent_t ev_b;
    if (!event(&ev_b) ||
        cudaMemcpy2DAsync(dB, n.ldb * es_a, B_host, n.ldb * es_a, n.b_cols * es_a, n.b_rows, cudaMemcpyHostToDevice,
                          ctx->copy_in) != cudaSuccess ||
        cudaEventRecord(ev_b, ctx->copy_in) != cudaSuccess || cudaStreamWaitEvent(comp, ev_b, 0) != cudaSuccess)
        return finish(TC_ERR_CUDA);
    for (int i = 0; i < nb; ++i) {
        const int64_t m0 = (int64_t)i * band, m1 = std::min<int64_t>(d->M, m0 + band);
        cudaEvent_t ev_in, ev_done;
        if (!event(&ev_in) || !event(&ev_done) || copy_a(m0, m1) != cudaSuccess ||
            (d->beta != 0.0f && copy_c(m0, m1, cudaMemcpyHostToDevice, ctx->copy_in) != cudaSuccess) ||
            cudaEventRecord(ev_in, ctx->copy_in) != cudaSuccess || cudaStreamWaitEvent(comp, ev_in, 0) != cudaSuccess)
            return finish(TC_ERR_CUDA);
        tc_gemm_desc db = *d;
        db.M = (int32_t)(m1 - m0);
        db.lda = (int32_t)n.lda;
        db.ldb = (int32_t)n.ldb;
        db.ldc = (int32_t)n.ldc;
        const void *Ab = d->transpose_a ? static_cast<const void *>(dA + m0 * es_a)
                                        : static_cast<const void *>(dA + m0 * n.lda * es_a);
        st = run(ctx, &db, Ab, dB, dC + m0 * n.ldc * es_c, 1, 0, 0, 0, ctx->def);
        if (st != TC_OK) return finish(st);
        if (cudaEventRecord(ev_done, comp) != cudaSuccess || cudaStreamWaitEvent(ctx->copy_out, ev_done, 0) != cudaSuccess ||
            copy_c(m0, m1, cudaMemcpyDeviceToHost, ctx->copy_out) != cudaSuccess)
            return finish(TC_ERR_CUDA);
    }
    return finish(TC_OK);
}

tc_status_t tc_gemm_validate(const tc_gemm_desc *d, const void *A, const void *B, const void *C)
{
    Norm n;
    return validate(d, A, B, C, 1, 0, 0, 0, &n);
}

tc_status_t tc_gemm_batched_validate(const tc_gemm_batched_desc *bd, const void *A, const void *B, const void *C)
{
    if (!bd) return TC_ERR_NULL;
    Norm n;
    return validate(&bd->base, A, B, C, bd->batch, bd->stride_a, bd->stride_b, bd->stride_c, &n);
}

tc_status_t tc_gemm_epilogue_validate(const tc_gemm_desc *d, const tc_epilogue *epi, const void *A, const void *B,
                                      const void *C)
{
    Norm n;
    tc_status_t st = validate(d, A, B, C, 1, 0, 0, 0, &n);
    if (st != TC_OK) return st;
    return validate_epilogue(d, n, epi, C);
}

tc_status_t tc_gemm_plan(const tc_gemm_desc *d, const void *A, const void *B, const void *C, int num_sms, char *buf,
                         size_t len)
{
    if (!buf || len == 0) return TC_ERR_NULL;
    buf[0] = '\0';
    Norm n;
    tc_status_t st = validate(d, A, B, C, 1, 0, 0, 0, &n);
    if (st != TC_OK) return st;
    Plan p;
    if ((st = make_plan(d, n, A, B, num_sms, &p)) != TC_OK) return st;
    std::snprintf(buf, len, "%s", p.name.c_str());
    return TC_OK;
}

tc_status_t tc_gemm_splitk_noalloc(const tc_gemm_desc *d, const void *A, const void *B, void *C, int split,
                                   void *cuda_stream)
{
    Norm n;
    tc_status_t st = validate(d, A, B, C, 1, 0, 0, 0, &n);
    if (st != TC_OK) return st;
    if (d->a_dtype == TC_F32) return TC_ERR_DTYPE;
    if (split < 0) return TC_ERR_DIM;
    if (!aligned16(A) || !aligned16(B) || n.lda % 8 != 0 || n.ldb % 8 != 0) return TC_ERR_ALIGN_UNSUPPORTED;

    constexpr int bn = 128;
    const int64_t tiles = cdiv(d->M, BM) * cdiv(d->N, bn);
    const int64_t num_kb = cdiv(d->K, BK);
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
        return TC_ERR_CUDA;
    int64_t S = split;
    if (S == 0) S = std::max<int64_t>(1, std::min<int64_t>(sms / std::max<int64_t>(tiles, 1), num_kb / 4));
    S = std::min<int64_t>(S, num_kb);
    if (S > 1 && tiles * S * BM * bn * (int64_t)sizeof(float) > (int64_t)NOALLOC_PARTIAL_BYTES)
        return TC_ERR_SCRATCH;
    if (tiles * S > INT32_MAX / 2) return TC_ERR_OVERFLOW;

    NoallocScratch scratch;
    if (noalloc_scratch(&scratch) != cudaSuccess) return TC_ERR_CUDA;
    // the TMA descriptor encoder, looked up until a lookup succeeds (a
    // failed first lookup, e.g. before any device was usable, is retried)
    static std::mutex enc_mu;
    static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> enc_fn{nullptr};
    PFN_cuTensorMapEncodeTiled_v12000 encoder = enc_fn.load(std::memory_order_acquire);
    if (!encoder) {
        std::lock_guard<std::mutex> g(enc_mu);
        encoder = enc_fn.load(std::memory_order_acquire);
        if (!encoder) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                    cudaSuccess &&
                q == cudaDriverEntryPointSuccess && fn) {
                encoder = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
                enc_fn.store(encoder, std::memory_order_release);
            } else {
                cudaGetLastError();
            }
        }
    }
    if (!encoder) return TC_ERR_CUDA;
    tc_ctx enc;                 // carries only the encoder for encode_map; owns nothing
    enc.encode = encoder;

    MmaLaunch L{};
    L.bn = bn;
    L.cg = 1;
    L.grid = (int)std::min<int64_t>(tiles * S, sms);
    MmaArgs &a = L.args;
    a.M = d->M;
    a.N = d->N;
    a.K = d->K;
    a.num_kb = (int)num_kb;
    a.tiles_m = (int)cdiv(d->M, BM);
    a.tiles_n = (int)cdiv(d->N, bn);
    a.tiles_per_batch = (int)tiles;
    a.batch = 1;
    a.seg0_tiles = (int)tiles;
    a.seg0_split = (int)S;
    a.seg1_split = 1;
    a.split_base = 0;
    a.total_units = (int)(tiles * S);
    a.group_m = 4;
    a.a_kmajor = !d->transpose_a;
    a.b_kmajor = d->transpose_b;
    const uint32_t fmt = d->a_dtype == TC_BF16 ? 1u : 0u;
    a.idesc = (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(!a.a_kmajor) << 15) |
              ((uint32_t)(!a.b_kmajor) << 16) | ((uint32_t)(bn >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
    a.alpha = d->alpha;
    a.beta = d->beta;
    a.C = C;
    a.ldc = n.ldc;
    a.c_dtype = d->c_dtype;
    const int64_t ec = (int64_t)elem_size(d->c_dtype);
    a.c_vec_ok = aligned16(C) && (n.ldc * ec) % 16 == 0;
    a.c_tma = a.c_vec_ok;
    a.ws = S > 1 ? scratch.partials : nullptr;
    a.status = scratch.status;
    a.timeout_ns = 4000000000ull + (unsigned long long)num_kb * 20000ull;

    bool ok = a.a_kmajor ? encode_map(&enc, &L.tmA, d->a_dtype, A, d->K, d->M, n.lda, false, 1, 0, 64, BM)
                         : encode_map(&enc, &L.tmA, d->a_dtype, A, d->M, d->K, n.lda, false, 1, 0, 64, 64);
    if (ok)
        ok = a.b_kmajor ? encode_map(&enc, &L.tmB, d->a_dtype, B, d->K, d->N, n.ldb, false, 1, 0, 64, bn)
                        : encode_map(&enc, &L.tmB, d->a_dtype, B, d->N, d->K, n.ldb, false, 1, 0, 64, 64);
    if (ok && a.c_tma)
        ok = encode_map(&enc, &L.tmC, d->c_dtype, C, d->N, d->M, n.ldc, false, 1, 0, 32, 32,
                        d->c_dtype == TC_F32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
    if (ok && a.ws)
        ok = encode_map(&enc, &L.tmW, TC_F32, a.ws, bn, tiles * S * BM, bn, false, 1, 0, 32, 32,
                        CU_TENSOR_MAP_SWIZZLE_128B);
    if (!ok) return TC_ERR_CUDA;

    cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
    // the status word must start at zero; the partial tiles are fully overwritten
    if (cudaMemsetAsync(scratch.status, 0, sizeof(unsigned), stream) != cudaSuccess) return TC_ERR_CUDA;
    if (launch_mma(L, stream) != cudaSuccess) return TC_ERR_CUDA;
    if (a.ws) {
        ReduceArgs r{};
        r.ws = a.ws;
        r.rows_per_tile = BM;
        r.bn = bn;
        r.first_tile = 0;
        r.ntiles = (int)tiles;
        r.S = (int)S;
        r.tiles_m = a.tiles_m;
        r.tiles_n = a.tiles_n;
        r.tiles_per_batch = a.tiles_per_batch;
        r.group_m = a.group_m;
        r.M = d->M;
        r.N = d->N;
        r.alpha = d->alpha;
        r.beta = d->beta;
        r.C = C;
        r.ldc = n.ldc;
        r.stride_c = 0;
        r.c_dtype = d->c_dtype;
        r.c_vec_ok = a.c_vec_ok;   // 16-byte vectors of 8 elements (two for fp32)
        r.status = scratch.status;
        if (launch_reduce(r, stream) != cudaSuccess) return TC_ERR_CUDA;
    }
    return TC_OK;
}

const char *tc_last_kernel(tc_ctx *ctx) { return ctx ? ctx->last.c_str() : ""; }

uint64_t tc_launch_count(tc_ctx *ctx) { return ctx ? ctx->launches : 0; }

}  // extern "C"
