// cpa_attn.cuh -- the paged attention kernel behind cascade verify (Pass A
// with fused Pass B + merge), Pass A alone, naive expand and prefix-hit
// prefill, for sm_103a.
//
// One persistent CTA per SM.  The key tiles of all work units are laid end to
// end and cut into one contiguous, equal-length range per CTA, so every SM
// streams the same number of KV bytes whatever the mix of sequence lengths.
// A unit whose tiles straddle two CTAs is finished by whichever CTA arrives
// last: each piece writes (o, lse) as a partial and the last one merges them
// in CTA order with the log-sum-exp identity, so results do not depend on
// arrival order.
//
// Work unit:   cascade / Pass A  one request b and one KV head: its
//                                topk*S draft tokens x G query heads share
//                                one read of the prefix (M = topk*S*G rows);
//              naive expand      one branch (b, k) and one KV head: S*G rows,
//                                the same prefix read again for every k;
//              prefill           one KV head and 128/G suffix tokens.
//
// Warp roles (warp index w, 16 warps):
//   w = 0      producer: walks the block table (page ids prefetched 32 boxes
//              ahead by the whole warp) and issues TMA loads of 128-B
//              swizzled K/V boxes (one copy per lane) into a ring of 128-key
//              stages; for units of two M tiles it also loads Q by TMA;
//   w = 2      (bf16) producer of the V halves, beside warp 0's K halves;
//   w = 3      MMA issuer (FP8 instance: w = 1, and w = 2, 3 widen the E4M3
//              rows to f16): S = Q K^T (M=128, N=128, K=128) into TMEM, then
//              O += P V (M=128, N=128, K=128) into TMEM.  With one M tile Q
//              sits in TMEM and both MMAs read their A operand from there;
//   w = 4..11  softmax: two warpgroups.  With one M tile they split each
//              tile's 128 columns and swap per-row maxima every tile; with
//              two M tiles each owns one.  A thread reads its S row from TMEM,
//              masks, exponentiates (base 2) and writes bf16 P back over the
//              S columns it came from, rescaling O only when the running max
//              grew by more than 2^8.  On a unit's last tile (its drafts, or
//              the causal diagonal) it also writes the bf16 residual of P and
//              PV runs twice, so rows that see few keys keep P to ~16 bits;
//   w = 12..15 epilogue: O / l, the merge of units split across CTAs, store;
//              with one M tile it also stages the next units' Q in TMEM.
// Verify units end with one extra tile holding the unit's own draft tokens
// (Pass B): branch k's drafts fill rows k*sb.. of that tile and the softmax
// applies the causal-within-branch mask, so Pass B and its merge with Pass A
// run inside the same online softmax on the tensor cores.
#pragma once
#include <type_traits>
#include <cstdint>

#include "cpa_device.cuh"
#include "cpa_types.h"

namespace cpa {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

// Timestamps of pipeline events, only in builds that define CPA_TRACE (the
// diagnostic build: `python -m cascade_paged_attention_gb300.build --trace`,
// whose cpa_trace_set_buffer points cpa_trace_buf at a caller's buffer);
// otherwise no code.  Buffer layout (64-bit words):
//   [4 CTAs][64 event rows][1024]  clock64 of event `ev` at tile/unit `idx`
//                                  for CTAs 0..3 (rows 0..62; row 63 holds
//                                  those CTAs' start and end clock64 and
//                                  %globaltimer at indices 0..3);
//   then kTraceCtaWords words per CTA at kTraceCtaBase + kTraceCtaWords * CTA:
//     0 start (%globaltimer, after scheduling), 1 end, 2 producer done
//     issuing, 3 MMA issuer done, 4 epilogue done, 5 tiles, 6 units.
#ifdef CPA_TRACE
static __device__ unsigned long long* cpa_trace_buf = nullptr;
constexpr int kTraceCtaBase = 4 * 64 * 1024;
constexpr int kTraceCtaWords = 8;
constexpr int kTraceStampRow = 63;
#define CPA_TRACE_EVENT(ev, idx)                                                  \
    do {                                                                          \
        if (cpa_trace_local && blockIdx.x < 4 && (ev) < kTraceStampRow &&         \
            (idx) < 1024)                                                         \
            cpa_trace_local[(blockIdx.x * 64 + (ev)) * 1024 + (idx)] = clock64(); \
    } while (0)
#define CPA_TRACE_CTA(slot, value)                                                      \
    do {                                                                                \
        if (cpa_trace_local)                                                            \
            cpa_trace_local[kTraceCtaBase + kTraceCtaWords * blockIdx.x + (slot)] = (value); \
    } while (0)
#else
#define CPA_TRACE_EVENT(ev, idx) \
    do {                         \
    } while (0)
#define CPA_TRACE_CTA(slot, value) \
    do {                           \
    } while (0)
#endif

struct AttnParams {
    CUtensorMap qmap;
    CUtensorMap kmap;
    CUtensorMap vmap;
    CUtensorMap kdmap;  // K/V pool with draft-block boxes (sb rows)
    CUtensorMap vdmap;
    const __nv_bfloat16* q;
    const __nv_bfloat16* k_pages;
    const __nv_bfloat16* v_pages;
    const int32_t* ptab;  // prefix table (verify) / sequence table (prefill)
    const int32_t* dtab;  // draft table (verify) / tree table (tree verify)
    const int32_t* tree_par;  // tree verify: [B][S] parent index of every node (-1: a root)
    const int32_t* lens;  // prefix lengths (verify)
    // verify over a prefix shared by groups of s_grp consecutive requests: the
    // first s_len logical positions (a whole number of pages) of request b are
    // the shared prefix of its group, read through row b / s_grp of stab; the
    // request's own prefix (lens[b] tokens, table ptab) follows it.  s_len = 0:
    // no shared segment.
    const int32_t* stab;
    int stab_stride, s_len, s_grp;
    void* o;
    float* lse;
    // when set, every finished row is merged with this partial result of the
    // same rows (fp32 o [T, H_q, 128], natural-log lse [T, H_q]) by the LSE
    // identity before it is written (multi-level verify: the shared level)
    const float* mrg_o;
    const float* mrg_lse;
    uint32_t* status;
    uint32_t* counters;
    // split-unit parts, one slot per (CTA, first or last piece): o as 32 float4
    // column groups of NUM_MT*128 rows each (a slot's part is contiguous), lse
    // in log2 units; slots are kMaxUnitRows rows apart
    float* part_o;    // [2*n_ctas][32][kMaxUnitRows] float4
    float* part_lse;  // [2*n_ctas][kMaxUnitRows]
    int mode;
    int B, topk, S, H_q, H_kv, G, P, num_pages;
    int ptab_stride, dtab_stride, max_len;
    int N, H_hit, M, QT;  // prefill
    int upg;              // verify: units per request
    int TS;               // query tokens per unit
    int TSB;              // query tokens per M tile
    int Rq;               // rows of one Q M-tile buffer (multiple of 8)
    int boxr;             // rows of one K/V TMA box
    int n_stages, n_qbufs;
    int has_draft;        // cascade / naive: the unit's drafts form its last tile
    int sb;               // rows per branch block in the draft tile (8 or 16)
    int nbr;              // branches per unit (cascade topk, naive 1)
    int out_f32;          // o is fp32 (a partial for a later merge) instead of bf16
    float scale_log2;     // sm_scale * log2(e)
    // FP8 E4M3 pools (the FP8 kernel instance only): K/V elements are code x
    // scale, the scale one value per tensor or one per (KV head, channel).
    // Codes are widened exactly to f16 (e4m3x2_to_f16x2); Q is staged as
    // q * k_scale in f16 and the output multiplied by v_scale per channel.
    const float* k_scale;
    const float* v_scale;
    int scale_per_channel;
    int fp8;
    uint32_t off_q, off_kv;
};

// ------------------------------------------------------------------ units
struct Unit {
    int b, h;
    int t0, ntok;     // query tokens [t0, t0 + ntok)
    int p0;           // prefill: suffix position of token t0
    int branch0;      // verify: first branch of the unit
    int lo, hi;       // keys [lo, hi) visible (prefill full/tri: hi of the last row)
    int valid_end;    // keys at or past this are not in the sequence
    int tile_base;    // first key tile
    int n_prefix;     // prefix tiles; tile n_prefix (verify) holds the unit's drafts
    int n_tiles;
    int resid_tile;   // tile that also sends P's bf16 residual through PV, or -1
    const int32_t* trow;
};

__device__ __forceinline__ bool is_verify(int mode) {
    return mode <= MODE_PASS_A || mode == MODE_TREE;
}

__device__ __forceinline__ int prefix_len(const AttnParams& p, int b) {
    int L = __ldg(p.lens + b);
    return (L < 0 ? 0 : (L > p.max_len ? p.max_len : L)) + p.s_len;
}

__device__ __forceinline__ void prefill_keys(const AttnParams& p, int p0, int ntok, int& lo,
                                             int& hi) {
    if (p.mode == MODE_PREFILL_RECT) {
        lo = 0;
        hi = p.H_hit;
    } else if (p.mode == MODE_PREFILL_TRI) {
        lo = p.H_hit;
        hi = p.H_hit + p0 + ntok;
    } else {
        lo = 0;
        hi = p.H_hit + p0 + ntok;
    }
}

__device__ __forceinline__ int tiles_for(int lo, int hi) {
    int t = (hi + kBN - 1) / kBN - lo / kBN;
    return t < 1 ? 1 : t;
}

__device__ __forceinline__ int prefill_qt_tiles(const AttnParams& p, int qt) {
    int p0 = qt * p.TS;
    int ntok = min(p.TS, p.M - p0);
    int lo, hi;
    prefill_keys(p, p0, ntok, lo, hi);
    return tiles_for(lo, hi);
}

// Tiles of one verify unit with prefix length L: the prefix tiles, then (for
// cascade / naive) one tile holding the unit's own draft tokens.  A unit
// always has at least one tile, so every row gets an output.
__device__ __forceinline__ int verify_prefix_tiles(const AttnParams& p, int L) {
    const int t = (L + kBN - 1) / kBN;
    return p.has_draft ? t : (t < 1 ? 1 : t);
}
__device__ __forceinline__ int verify_unit_tiles(const AttnParams& p, int L) {
    return verify_prefix_tiles(p, L) + (p.has_draft ? 1 : 0);
}

// P goes through the tensor cores in bf16.  Over many keys its rounding errors
// average out; when a unit has few keys they do not, and the output would carry
// up to 2^-9 of |v| on top of its own bf16 rounding.  So a small unit's last
// tile (the one holding every key of the rows that see the fewest) also sends
// what the rounding dropped, itself in bf16, through a second PV pass.
constexpr int kResidMaxKeys = 512;

__device__ __forceinline__ Unit get_unit(const AttnParams& p, int u) {
    Unit x;
    if (is_verify(p.mode)) {
        const int b = u / p.upg, rem = u % p.upg;
        const int L = prefix_len(p, b);
        x.b = b;
        x.lo = 0;
        x.hi = L;
        x.valid_end = L;
        x.tile_base = 0;
        x.n_prefix = verify_prefix_tiles(p, L);
        x.n_tiles = verify_unit_tiles(p, L);
        x.p0 = 0;
        x.trow = p.ptab + (size_t)b * p.ptab_stride;
        if (p.mode == MODE_NAIVE) {
            const int k = rem / p.H_kv;
            x.h = rem % p.H_kv;
            x.branch0 = k;
            x.t0 = (b * p.topk + k) * p.S;
            x.ntok = p.S;
        } else {
            x.h = rem;
            x.branch0 = 0;
            x.t0 = b * p.TS;
            x.ntok = p.TS;
        }
    } else {
        const int grp = u / p.QT, qt = u % p.QT;
        x.b = grp / p.H_kv;
        x.h = grp % p.H_kv;
        x.p0 = qt * p.TS;
        x.ntok = min(p.TS, p.M - x.p0);
        x.t0 = x.b * p.M + x.p0;
        x.valid_end = p.N;
        x.branch0 = 0;
        prefill_keys(p, x.p0, x.ntok, x.lo, x.hi);
        x.tile_base = x.lo / kBN;
        x.n_tiles = tiles_for(x.lo, x.hi);
        x.n_prefix = x.n_tiles;
        x.trow = p.ptab + (size_t)x.b * p.ptab_stride;
    }
    // (f16 P in the FP8 kernel keeps 11 bits: no residual pass there)
    x.resid_tile = !p.fp8 && (x.hi - x.lo) + (p.has_draft ? p.S : 0) <= kResidMaxKeys
                       ? x.n_tiles - 1
                       : -1;
    return x;
}


// ------------------------------------------------------------------ shared control block
struct Ctrl {
    uint64_t kv_full[4], kv_empty[4];
    uint64_t q_full[2], q_empty[2];
    uint64_t s_full[2], p_full[2], p_empty[2];
    uint64_t o_full, o_empty, stats_full;
    uint64_t mma_done;
    uint64_t merge_full;  // other CTAs' parts of a split unit staged for the merge
    uint64_t cv_full[4];   // FP8: the stage's K codes are widened to f16
    uint64_t cvv_full[4];  // FP8: the stage's V codes are widened to f16
    // FP8: bit r of vrows[stage][r / 32]: V row r of the stage's tile holds a key
    // of the sequence (loaded, before the end); other V rows are zeroed
    uint32_t vrows[4][4];
    uint32_t tmem_base;
    uint32_t abort_flag;
    int64_t total;   // tiles of the whole problem
    int64_t begin;   // this CTA's first tile
    int64_t count;   // this CTA's tiles
    int64_t ustart;  // global tile index where the first unit starts
    int n_ctas;      // CTAs that have work
    int u0, j0;      // first unit and its first tile
    int rr, ppg, qtn;  // prefill: pairs dealt round-robin, pairs per group, q tiles per group
    int flag;
    int found;
    long long scan[32];
};
static_assert(sizeof(Ctrl) <= 1024, "control block");

constexpr uint32_t kOffStats = 1024;  // float2 [256]: (max, sum) per row of a finished unit
constexpr uint32_t kOffXchg = 3072;   // float [2][2][128]: per-half row maxima, by tile parity
constexpr uint32_t kOffSum = 5120;    // float [128]: second half's row sums at a unit's end
constexpr uint32_t kOffData = 6144;   // first 1024-aligned byte after the above
constexpr uint32_t kStageBytes = 4u * kBN * 128u;  // K lo/hi, V lo/hi halves: 64 KB

// Per-configuration layout.  NUM_MT = 1: units of up to 128 rows; Q lives in
// TMEM (S = Q K^T reads its A operand from TMEM) and two softmax warpgroups
// split each tile's 128 columns.  NUM_MT = 2: units of up to 256 rows in two
// M tiles; Q lives in shared memory and each softmax warpgroup owns an M tile.
template <int NUM_MT>
struct Cfg {
    static constexpr bool kQInTmem = NUM_MT == 1;
    static constexpr int kSplit = NUM_MT == 1 ? 2 : 1;  // softmax warpgroups per M tile
    static constexpr int kSBufs = NUM_MT == 1 ? 2 : 1;  // S buffers per M tile
    static constexpr int kSmWarp0 = 4;                   // 8 softmax warps: 4..11
    static constexpr int kEpiWarp0 = 12;                 // 4 epilogue warps: 12..15
    static constexpr int kThreads = 512;
    static constexpr uint32_t kTmemCols = 512;
    // TMEM columns.  Q (bf16, 2 per column): 64 per buffer; S: 128 per buffer
    // (the P of each 64-key half overwrites the first 32 of that half's S
    // columns, its residual the other 32); O: 128.
    static constexpr uint32_t q_col(int qb) { return (uint32_t)qb * 64u; }
    static constexpr uint32_t s_col(int mt, int sb) {
        return (kQInTmem ? 128u : 0u) + (uint32_t)(mt * kSBufs + sb) * 128u;
    }
    static constexpr uint32_t o_col(int mt) {
        return (kQInTmem ? 128u : 0u) + (uint32_t)(NUM_MT * kSBufs) * 128u + (uint32_t)mt * 128u;
    }
    static_assert((kQInTmem ? 128 : 0) + NUM_MT * kSBufs * 128 + NUM_MT * 128 <= 512,
                  "TMEM columns");
};

// Inclusive block-wide prefix sum of one int64 per thread; returns the
// exclusive prefix and the block total.
__device__ __forceinline__ long long block_scan(long long v, long long* ws, long long& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    long long x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) ws[warp] = x;
    __syncthreads();
    if (warp == 0) {
        long long w = lane < nw ? ws[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            long long y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        ws[lane] = w;
    }
    __syncthreads();
    const long long base = warp > 0 ? ws[warp - 1] : 0;
    total = ws[nw - 1];
    __syncthreads();
    return base + x - v;
}

// Every thread of the CTA: find the problem's total tile count and where this
// CTA's range begins.
template <bool FAST32>
__device__ __forceinline__ void schedule(const AttnParams& p, Ctrl* c) {
    long long total = 0;
    const int nthr = blockDim.x;
    if (is_verify(p.mode)) {
        // group = request; every unit of a request has the same tile count
        for (int b0 = 0; b0 < p.B; b0 += nthr) {
            const int b = b0 + threadIdx.x;
            long long v = 0;
            if (b < p.B) {
                const int L = __ldg(p.lens + b);
                if (L < 0 || L > p.max_len) atomicOr(p.status, CPA_DEV_BAD_LENGTH);
                v = (long long)p.upg * verify_unit_tiles(p, prefix_len(p, b));
            }
            long long tot;
            block_scan(v, c->scan, tot);
            total += tot;
        }
    } else if (p.mode == MODE_PREFILL_RECT) {
        // rectangle only: every unit reads the same keys 0..H-1, so units are of
        // equal size and are split contiguously like verify units
        total = (long long)p.B * p.H_kv * p.QT * tiles_for(0, p.H_hit);
    } else {
        // Prefill: every q tile of a group (request, KV head) reads the same keys
        // from the start, so the work is dealt so that the CTAs running at any one
        // time work on the same groups and share each K/V tile through L2: the
        // pairs (q tile j, q tile QT-1-j) of a group, which have equal tile sums,
        // go round-robin over the CTAs in group order.  Units are never split.
        if (threadIdx.x == 0) {
            const int ppg = (p.QT + 1) / 2;
            const long long pairs = (long long)p.B * p.H_kv * ppg;
            const int n = (int)(pairs < (long long)gridDim.x ? pairs : (long long)gridDim.x);
            const int cta = blockIdx.x;
            c->rr = 1;
            c->ppg = ppg;
            c->qtn = p.QT;
            c->n_ctas = n;
            c->total = 0;
            c->found = 1;
            long long cnt = 0;
            for (long long pid = cta; pid < pairs && cta < n; pid += n) {
                const int jp = (int)(pid % ppg);
                cnt += prefill_qt_tiles(p, jp);
                if (p.QT - 1 - jp != jp) cnt += prefill_qt_tiles(p, p.QT - 1 - jp);
            }
            c->count = cnt;
            c->begin = 0;
            c->u0 = (int)((cta / ppg) * p.QT + cta % ppg);
            c->j0 = 0;
            c->ustart = cta;  // the pair this CTA starts with
        }
        __syncthreads();
        return;
    }
    const int n_ctas = (int)(total < (long long)gridDim.x ? total : (long long)gridDim.x);
    const int cta = blockIdx.x;
    if (threadIdx.x == 0) {
        c->rr = 0;
        c->total = total;
        c->n_ctas = n_ctas;
        c->found = 0;
        if (cta < n_ctas) {
            c->begin = split_begin(total, n_ctas, cta, FAST32);
            c->count = split_begin(total, n_ctas, cta + 1, FAST32) - c->begin;
        } else {
            c->begin = 0;
            c->count = 0;
        }
    }
    __syncthreads();
    if (c->count == 0) return;
    const long long t0 = c->begin;
    if (is_verify(p.mode)) {
        long long run = 0;
        for (int b0 = 0; b0 < p.B; b0 += nthr) {
            const int b = b0 + threadIdx.x;
            long long v = 0;
            int tpu = 1;
            if (b < p.B) {
                tpu = verify_unit_tiles(p, prefix_len(p, b));
                v = (long long)p.upg * tpu;
            }
            long long tot;
            const long long ex = block_scan(v, c->scan, tot);
            if (b < p.B && run + ex <= t0 && t0 < run + ex + v) {
                const long long off = t0 - (run + ex);
                c->u0 = b * p.upg + (int)(off / tpu);
                c->j0 = (int)(off % tpu);
                c->ustart = run + ex + (off / tpu) * tpu;
                c->found = 1;
            }
            run += tot;
            __syncthreads();
            if (c->found) break;
        }
    } else if (threadIdx.x == 0) {
        const int tpu = tiles_for(0, p.H_hit);
        c->u0 = (int)(t0 / tpu);
        c->j0 = (int)(t0 % tpu);
        c->ustart = (t0 / tpu) * tpu;
        c->found = 1;
    }
    __syncthreads();
}

// Walks this CTA's tiles unit by unit; every role runs its own copy.
struct Walker {
    int u, j;
    long long ustart;
    long long left;
    int seg;
    __device__ __forceinline__ void init(const Ctrl* c) {
        u = c->u0;
        j = c->j0;
        ustart = c->ustart;
        left = c->count;
        seg = 0;
    }
    // Tiles [jb, je) of unit x that belong to this CTA.
    __device__ __forceinline__ void piece(const Unit& x, int& jb, int& je) const {
        jb = j;
        const long long rest = (long long)x.n_tiles - j;
        je = (int)(j + (left < rest ? left : rest));
    }
    __device__ __forceinline__ void next(const Unit& x, int jb, int je, const Ctrl* c) {
        left -= (je - jb);
        j = 0;
        ++seg;
        if (!c->rr) {
            ustart += x.n_tiles;
            ++u;
            return;
        }
        // round-robin prefill: ustart is the current pair
        const int QT = c->qtn, pid = (int)ustart, jp = pid % c->ppg;
        if (u % QT == jp && QT - 1 - jp != jp) {
            u += QT - 1 - 2 * jp;  // the pair's second q tile
        } else {
            const int nxt = pid + c->n_ctas;
            ustart = nxt;
            u = (nxt / c->ppg) * QT + nxt % c->ppg;
        }
    }
};

// A tile-by-tile cursor over this CTA's range: the unit, the tile within it,
// and whether the tile opens or closes this CTA's piece of the unit.
struct TileCursor {
    Walker w;
    Unit x;
    int jb, je, jj;
    __device__ __forceinline__ void init(const Ctrl* c, const AttnParams& p) {
        w.init(c);
        if (w.left > 0) {
            x = get_unit(p, w.u);
            w.piece(x, jb, je);
            jj = jb;
        }
    }
    __device__ __forceinline__ bool first() const { return jj == jb; }
    __device__ __forceinline__ bool last() const { return jj == je - 1; }
    __device__ __forceinline__ void advance(const AttnParams& p, const Ctrl* c) {
        if (++jj == je) {
            w.next(x, jb, je, c);
            if (w.left > 0) {
                x = get_unit(p, w.u);
                w.piece(x, jb, je);
                jj = jb;
            }
        }
    }
};

// ------------------------------------------------------------------ epilogue helpers
__device__ __forceinline__ void named_bar_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Kernel variants.  Each is a separate instance so that the common paths
// carry no extra code (and no extra registers).
enum Variant : int {
    VAR_PLAIN = 0,  // bf16 pools
    VAR_FP8 = 1,    // FP8 E4M3 pools, widened on chip (one M tile)
    VAR_TREE = 2,   // tree verify: the unit's last tile holds the draft tree,
                    // masked per row by ancestor masks
    VAR_MERGE = 3,  // bf16 pools; every finished row is merged with another
                    // launch's partial result (p.mrg_o) before it is written
    VAR_PREFILL = 4,  // prefill (full or triangle): units are never split and
                      // have no draft tile, so neither path is compiled in
};

template <int NUM_MT, int VAR>
__global__ void __launch_bounds__(Cfg<NUM_MT>::kThreads, 1)
    paged_attn_kernel(const __grid_constant__ AttnParams p) {
    using C = Cfg<NUM_MT>;
    constexpr int kPartRows = NUM_MT * 128;  // rows of a split-unit part (see part_o)
    constexpr bool FP8 = VAR == VAR_FP8;
    constexpr bool TREE = VAR == VAR_TREE;
    // 32-bit division in the work split: faster in every instance but the tree
    // one, which measured 112.7 us without it against 117.4 us with it
    constexpr bool kFast32 = !TREE;
    constexpr bool MERGE = VAR == VAR_MERGE;
    constexpr bool PREFILL = VAR == VAR_PREFILL;
#ifdef CPA_TRACE
    unsigned long long* const cpa_trace_local = cpa_trace_buf;  // read once
#endif
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Ctrl* ctrl = reinterpret_cast<Ctrl*>(smem);
    float2* stats = reinterpret_cast<float2*>(smem + kOffStats);
    float* xchg = reinterpret_cast<float*>(smem + kOffXchg);
    float* xsum = reinterpret_cast<float*>(smem + kOffSum);
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // The thread that issues the MMAs shares its SMSP (warp % 4) with the two
    // softmax warps of TMEM lanes 32 (warp % 4) .. +31.  Warp 3 puts it beside
    // the warps of rows 96..127, which have nothing to do in units of up to 96
    // rows (the verify shapes): 1-2 % faster there than beside rows 32..63.  The
    // FP8 instance widens on warps 2 and 3 and issues from warp 1.
    constexpr int kMmaWarp = FP8 ? 1 : 3;
    volatile uint32_t* abort_flag = &ctrl->abort_flag;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 4; ++i) {
            mbar_init(&ctrl->kv_full[i], FP8 ? 1 : 2);  // one arrival per producer warp
            mbar_init(&ctrl->kv_empty[i], 1);
            mbar_init(&ctrl->cv_full[i], 2);  // the two widening warps
            mbar_init(&ctrl->cvv_full[i], 2);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ctrl->q_full[i], C::kQInTmem ? 4 : 1);  // 4 epilogue warps / the TMA
            mbar_init(&ctrl->q_empty[i], 1);
            mbar_init(&ctrl->s_full[i], 1);
            mbar_init(&ctrl->p_full[i], 4 * C::kSplit);  // the warps writing that P
            mbar_init(&ctrl->p_empty[i], 1);
        }
        mbar_init(&ctrl->o_full, 1);
        // one arrival per warp (after __syncwarp): arrivals of every thread would
        // serialise on the barrier's word
        mbar_init(&ctrl->o_empty, 4);
        mbar_init(&ctrl->stats_full, 4 * NUM_MT);
        mbar_init(&ctrl->mma_done, 1);
        mbar_init(&ctrl->merge_full, 1);
        ctrl->abort_flag = 0;
        fence_barrier_init();
        prefetch_tmap(&p.kmap);
        prefetch_tmap(&p.vmap);
        if (!C::kQInTmem) prefetch_tmap(&p.qmap);
    }
    if (warp == 1) {
        tmem_alloc(&ctrl->tmem_base, C::kTmemCols);
        tmem_relinquish();
    }
    // V rows a tile does not load (past a sequence's end, past a branch's drafts)
    // keep what an earlier tile left there; zero every V stage once so that this
    // is always finite data, which P = 0 multiplies away
    for (int i = threadIdx.x; i < p.n_stages * 2 * kBN * 8; i += blockDim.x) {
        const int st = i / (2 * kBN * 8), rem = i % (2 * kBN * 8);
        *reinterpret_cast<uint4*>(smem + p.off_kv + st * kStageBytes + 2 * kBN * 128 + rem * 16) =
            make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    schedule<kFast32>(p, ctrl);
#ifdef CPA_TRACE
    if (threadIdx.x == 0 && cpa_trace_local) {
        if (blockIdx.x < 4) {
            cpa_trace_local[(blockIdx.x * 64 + kTraceStampRow) * 1024 + 0] = clock64();
            cpa_trace_local[(blockIdx.x * 64 + kTraceStampRow) * 1024 + 1] = globaltimer_ns();
        }
        CPA_TRACE_CTA(0, globaltimer_ns());
        CPA_TRACE_CTA(5, (unsigned long long)ctrl->count);
    }
#endif
    const uint32_t tmem = ctrl->tmem_base;
    const int n_ctas = ctrl->n_ctas;
    const long long total = ctrl->total;
    const int G = p.G;

    if (ctrl->count > 0) {
        if (warp == 0 || (!FP8 && warp == 2)) {
            // ============================== producers
            // bf16: warp 0 loads the K halves of every box and warp 2 the V halves
            // (two warps issue TMA copies faster than one); FP8: warp 0 loads both.
            // verify reads each K/V tile once; prefill reads it once per q tile
            const uint64_t pol_kv =
                is_verify(p.mode) ? l2_policy_evict_first() : l2_policy_evict_normal();
            const uint64_t pol_q = l2_policy_evict_last();
            const int NB = kBN / p.boxr;
            // TMA copies per box: bf16 K lo/hi and V lo/hi halves (64 columns x
            // 128 B rows each); FP8 K and V (128 one-byte columns, 128 B rows),
            // which land in the hi-half regions and are widened in place.
            // Every copy moves 128 B per row.
            constexpr int kParts = FP8 ? 2 : 4;
            auto region = [](int part) { return FP8 ? 2 * part + 1 : part; };
            auto col0 = [](int part) { return FP8 ? 0 : (part & 1) * 64; };
            // this warp's copies: parts [kPP * pi, kPP * pi + kPP) of every box
            constexpr int kPP = FP8 ? kParts : kParts / 2;
            const int pi = warp == 0 ? 0 : 1;
            const uint32_t q_tx = (uint32_t)(NUM_MT * 2 * G * p.TSB * 128);
            const uint32_t qmt_bytes = (uint32_t)(2 * p.Rq * 128);
            Walker w;
            w.init(ctrl);
            long long g = 0;
            int pst = 0;          // stage of tile g
            uint32_t pkpar = 0;   // parity of that stage's current use
            bool ok = true;
            while (w.left > 0 && ok) {
                const Unit x = get_unit(p, w.u);
                int jb, je;
                w.piece(x, jb, je);
                if (!C::kQInTmem && pi == 0) {
                    const int qb = w.seg % p.n_qbufs;
                    if (w.seg >= p.n_qbufs)
                        ok = mbar_wait_warp(&ctrl->q_empty[qb], ((w.seg / p.n_qbufs) - 1) & 1,
                                            abort_flag, p.status);
                    if (!ok) break;
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&ctrl->q_full[qb], q_tx);
                        for (int mt = 0; mt < NUM_MT; ++mt) {
                            uint8_t* dst = smem + p.off_q + (qb * NUM_MT + mt) * qmt_bytes;
                            const int tok = x.t0 + mt * p.TSB;
                            tma_load_3d(dst, &p.qmap, 0, x.h * G, tok, &ctrl->q_full[qb], pol_q);
                            tma_load_3d(dst + p.Rq * 128, &p.qmap, 64, x.h * G, tok,
                                        &ctrl->q_full[qb], pol_q);
                        }
                    }
                }
                // block-table window: lane l holds the page of box (wbase + l)
                const int key_base = x.tile_base * kBN;
                auto load_page = [&](int box) -> int {
                    const int pos = key_base + box * p.boxr;
                    if (pos >= x.valid_end) return -1;
                    if (pos < p.s_len)  // the group's shared prefix
                        return __ldg(p.stab + (size_t)(x.b / p.s_grp) * p.stab_stride + pos / p.P);
                    return __ldg(x.trow + (pos - p.s_len) / p.P);
                };
                int wbase = jb * NB;
                int cur = load_page(wbase + lane);
                int nxt = load_page(wbase + 32 + lane);
                // first draft page of branch `lane`, if this piece ends with the draft tile
                int dpage = -1;
                if (!TREE && p.has_draft && je == x.n_tiles && lane < p.nbr)
                    dpage = __ldg(p.dtab + (size_t)(x.b * p.topk + x.branch0 + lane) * p.dtab_stride);
                for (int jj = jb; jj < je; ++jj, ++g) {
                    // stage st of the ring, used for the (k+1)-th time; its previous use
                    // had parity kpar ^ 1 (kept incrementally: no 64-bit division here)
                    const int st = pst;
                    if (g >= p.n_stages) {
                        ok = mbar_wait_warp(&ctrl->kv_empty[st], pkpar ^ 1u, abort_flag, p.status);
                        if (!ok) break;
                    }
                    if (++pst == p.n_stages) {
                        pst = 0;
                        pkpar ^= 1u;
                    }
                    if (lane == 0) CPA_TRACE_EVENT(0, g);
                    uint8_t* stage = smem + p.off_kv + st * kStageBytes;
                    if (TREE && jj >= x.n_prefix) {
                        // the unit's tree tile: node j (j < S = N) is at logical position j
                        // of the request's tree table, row j of the tile; box bi = lane
                        const int32_t* ttab = p.dtab + (size_t)x.b * p.dtab_stride;
                        const int tpos = lane * p.boxr;
                        bool use = lane < NB && tpos < p.S;
                        const int tpg = use ? __ldg(ttab + tpos / p.P) : -1;
                        if (use && (tpg < 0 || tpg >= p.num_pages)) {
                            atomicOr(p.status, CPA_DEV_BAD_PAGE);
                            use = false;
                        }
                        const uint32_t mask = __ballot_sync(0xffffffffu, use);
                        if (lane == 0)
                            mbar_arrive_expect_tx(&ctrl->kv_full[st],
                                                  (uint32_t)__popc(mask) * kPP * p.boxr * 128u);
                        __syncwarp();
                        for (int t0 = 0; t0 < kPP * NB; t0 += 32) {
                            const int t = t0 + lane;
                            const int bi = (t < kPP * NB ? t : 0) / kPP;
                            const int part = kPP * pi + t % kPP;
                            const int pgi = __shfl_sync(0xffffffffu, tpg, bi & 31);
                            if (t < kPP * NB && (mask >> bi & 1u))
                                tma_load_3d(stage + region(part) * (kBN * 128) + bi * p.boxr * 128,
                                            part < kParts / 2 ? &p.kmap : &p.vmap, col0(part), x.h,
                                            pgi * p.P + ((bi * p.boxr) & (p.P - 1)),
                                            &ctrl->kv_full[st], pol_kv);
                        }
                        continue;
                    }
                    if (!PREFILL && jj >= x.n_prefix) {
                        // the unit's draft tile: branch k's drafts 0..S-1 sit in slots
                        // 0..S-1 of its first draft page; copy t = 4k + part loads one
                        // sb-row box (K lo/hi, V lo/hi) into rows k*sb.. of the tile
                        bool use = lane < p.nbr;
                        if (use && (dpage < 0 || dpage >= p.num_pages)) {
                            atomicOr(p.status, CPA_DEV_BAD_PAGE);
                            use = false;
                        }
                        const uint32_t mask = __ballot_sync(0xffffffffu, use);
                        if (FP8 && lane == 0) {
                            // rows k*sb .. k*sb+S-1 of every loaded branch k
                            uint32_t vr[4] = {0u, 0u, 0u, 0u};
                            for (int k = 0; k < p.nbr; ++k)
                                if (mask >> k & 1u)
                                    for (int s2 = 0; s2 < p.S; ++s2) {
                                        const int r = k * p.sb + s2;
                                        vr[r >> 5] |= 1u << (r & 31);
                                    }
                            for (int i = 0; i < 4; ++i) ctrl->vrows[st][i] = vr[i];
                        }
                        if (lane == 0)
                            mbar_arrive_expect_tx(&ctrl->kv_full[st],
                                                  (uint32_t)__popc(mask) * kPP * p.S * 128u);
                        __syncwarp();
                        // every lane runs the same iterations (the shuffle needs the whole
                        // warp); only the copy itself is predicated
                        for (int t0 = 0; t0 < kPP * p.nbr; t0 += 32) {
                            const int t = t0 + lane;
                            const int k = (t < kPP * p.nbr ? t : 0) / kPP;
                            const int part = kPP * pi + t % kPP;
                            const int pg = __shfl_sync(0xffffffffu, dpage, k & 31);
                            if (t < kPP * p.nbr && (mask >> k & 1u))
                                tma_load_3d(stage + region(part) * (kBN * 128) + k * p.sb * 128,
                                            part < kParts / 2 ? &p.kdmap : &p.vdmap, col0(part),
                                            x.h, pg * p.P, &ctrl->kv_full[st], pol_kv);
                        }
                        continue;
                    }
                    const int box0 = jj * NB;
                    if (box0 >= wbase + 32) {
                        cur = nxt;
                        wbase += 32;
                        nxt = load_page(wbase + 32 + lane);
                    }
                    const int my_box = box0 + (lane < NB ? lane : 0);
                    int pg = __shfl_sync(0xffffffffu, cur, (my_box - wbase) & 31);
                    const int pos = key_base + my_box * p.boxr;
                    bool use = lane < NB && pos < x.valid_end;
                    if (use && (pg < 0 || pg >= p.num_pages)) {
                        atomicOr(p.status, CPA_DEV_BAD_PAGE);
                        use = false;
                    }
                    const uint32_t mask = __ballot_sync(0xffffffffu, use);
                    if (FP8) {
                        // row r holds a key when its box was loaded and it is before the end
                        const int key0 = key_base + box0 * p.boxr;
                        const int boxr_log2 = 31 - __clz(p.boxr);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int r = 32 * i + lane;
                            const uint32_t v = __ballot_sync(
                                0xffffffffu, (mask >> (r >> boxr_log2) & 1u) && key0 + r < x.valid_end);
                            if (lane == 0) ctrl->vrows[st][i] = v;
                        }
                    }
                    if (lane == 0)
                        mbar_arrive_expect_tx(&ctrl->kv_full[st],
                                              (uint32_t)__popc(mask) * kPP * p.boxr * 128u);
                    __syncwarp();
                    // One TMA per lane: a thread issues its TMA copies one after another,
                    // so the kPP*NB copies of this warp are spread over the lanes.  Copy
                    // t loads part kPP*pi + t%kPP of box t/kPP.  Every lane runs the same
                    // iterations (the shuffle needs the whole warp).
                    for (int t0 = 0; t0 < kPP * NB; t0 += 32) {
                        const int t = t0 + lane;
                        const int bi = (t < kPP * NB ? t : 0) / kPP;
                        const int part = kPP * pi + t % kPP;
                        const int pgi = __shfl_sync(0xffffffffu, pg, bi & 31);
                        if (t < kPP * NB && (mask >> bi & 1u)) {
                            const int posi = key_base + (box0 + bi) * p.boxr;
                            tma_load_3d(stage + region(part) * (kBN * 128) + bi * p.boxr * 128,
                                        part < kParts / 2 ? &p.kmap : &p.vmap, col0(part), x.h,
                                        pgi * p.P + (posi & (p.P - 1)), &ctrl->kv_full[st], pol_kv);
                        }
                    }
                }
                w.next(x, jb, je, ctrl);
            }
            if (lane == 0) CPA_TRACE_CTA(2, globaltimer_ns());
            // make sure no TMA write is still in flight when the CTA leaves
            const long long filled = g;
            for (int st = 0; st < p.n_stages; ++st) {
                if (st < filled) {
                    const long long last = st + ((filled - 1 - st) / p.n_stages) * p.n_stages;
                    mbar_wait(&ctrl->kv_full[st], (uint32_t)((last / p.n_stages) & 1), abort_flag,
                              p.status);
                }
            }
        } else if (warp == kMmaWarp) {
            // ============================== MMA issuer
            // The work is a sequence of items, one per (tile, M tile): item i uses S
            // buffer i % 2 (one M tile: consecutive tiles alternate between two S
            // buffers; two M tiles: each M tile has its own).  Two cursors walk the
            // items: one issues S = Q K^T as soon as an item's K/V and Q are in place
            // and its S buffer is free (PV of item i - 2 issued), the other O += P V
            // as soon as the softmax has written that item's P.  Whichever is ready
            // goes first, so with two M tiles the tensor core works on one M tile
            // while the softmax works on the other.
            if (lane == 0) {
                // FP8 pools: every operand is f16 (Q, the widened K/V, P)
                const uint32_t idesc_s =
                    FP8 ? idesc_f16_f32(128, kBN, false) : idesc_bf16_f32(128, kBN, false);
                const uint32_t idesc_o =
                    FP8 ? idesc_f16_f32(128, 128, true) : idesc_bf16_f32(128, 128, true);
                // the stage is ready for the MMAs when it has landed (bf16) or has
                // also been widened (FP8); both barriers complete once per use
                uint64_t* const ready = FP8 ? ctrl->cv_full : ctrl->kv_full;
                const uint32_t qmt_bytes = (uint32_t)(2 * p.Rq * 128);
                TileCursor cs, cp;
                cs.init(ctrl, p);
                cp.init(ctrl, p);
                long long is = 0, ip = 0;  // next item for S / for PV
                const long long n_items = ctrl->count * NUM_MT;
                // K/V stage and kv_full parity of the tile S is at, and the stage of the
                // tile PV is at, kept incrementally (no 64-bit division in this loop)
                int st_s = 0, st_p = 0;
                uint32_t par_s = 0, par_p = 0;
                uint64_t t_idle = 0;
                uint32_t spins = 0;
                bool ok = true;
                while (ip < n_items) {
                    bool progressed = false;
                    // With two M tiles, PV of an item is issued before S of the next when
                    // both are ready (it frees the stage sooner: 442 -> 426 us on the
                    // long/variable workload); with one M tile S goes first (1 us better)
                    auto try_s = [&]() {
                        if (is < n_items && is <= ip + 1) {
                            const long long gs = is / NUM_MT;
                            const int mt = (int)(is % NUM_MT);
                            const int qb = p.n_qbufs == 2 ? (cs.w.seg & 1) : 0;
                            const uint32_t qpar =
                                (uint32_t)((p.n_qbufs == 2 ? cs.w.seg >> 1 : cs.w.seg) & 1);
                            const int st = st_s;
                            const bool q_ready = !cs.first() || mbar_test(&ctrl->q_full[qb], qpar);
                            if (q_ready && mbar_test(&ready[st], par_s)) {
                                if (mt == 0) CPA_TRACE_EVENT(2, gs);
                                tc_fence_after_sync();
                                const int sb = (int)(is & 1);
                                const uint32_t kb = sbase + p.off_kv + st * kStageBytes;
                                const uint32_t qa = sbase + p.off_q + (qb * NUM_MT + mt) * qmt_bytes;
                                const uint32_t sd = tmem + C::s_col(0, 0) + (uint32_t)sb * 128u;
    #pragma unroll
                                for (int kk = 0; kk < 8; ++kk) {
                                    const uint64_t bd =
                                        sdesc_sw128(kb + (kk >> 2) * kBN * 128 + (kk & 3) * 32, 16, 1024);
                                    if (C::kQInTmem) {
                                        umma_bf16_ts(sd, tmem + C::q_col(qb) + kk * 8, bd, idesc_s,
                                                     kk > 0 ? 1u : 0u);
                                    } else {
                                        const uint64_t ad = sdesc_sw128(
                                            qa + (kk >> 2) * p.Rq * 128 + (kk & 3) * 32, 16, 1024);
                                        umma_bf16_ss(sd, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
                                    }
                                }
                                umma_commit(&ctrl->s_full[sb]);
                                if (mt == NUM_MT - 1) {
                                    if (cs.last()) umma_commit(&ctrl->q_empty[qb]);
                                    CPA_TRACE_EVENT(15, gs);
                                    cs.advance(p, ctrl);
                                    if (++st_s == p.n_stages) {
                                        st_s = 0;
                                        par_s ^= 1u;
                                    }
                                }
                                ++is;
                                progressed = true;
                            }
                        }
                    };
                    auto try_pv = [&]() {
                        if (ip < is) {
                            const long long gp = ip / NUM_MT;
                            const int mt = (int)(ip % NUM_MT);
                            const int sb = (int)(ip & 1);
                            bool ready = mbar_test(&ctrl->p_full[sb], (uint32_t)((ip >> 1) & 1));
                            if (FP8 && ready) ready = mbar_test(&ctrl->cvv_full[st_p], par_p);
                            if (ready && cp.first() && cp.w.seg >= 1)
                                ready = mbar_test(&ctrl->o_empty, (uint32_t)((cp.w.seg - 1) & 1));
                            if (ready) {
                                if (mt == 0) CPA_TRACE_EVENT(3, gp);
                                tc_fence_after_sync();
                                const int st = st_p;
                                const uint32_t vb = sbase + p.off_kv + st * kStageBytes + 2 * kBN * 128;
                                const bool first = cp.first();
                                const int passes = cp.jj == cp.x.resid_tile ? 2 : 1;
                                // P of keys 64c..64c+63 (bf16, two per column) sits in the
                                // first 32 of the 64 S columns those keys came from, its
                                // residual in the other 32
                                const uint32_t pa = tmem + C::s_col(0, 0) + (uint32_t)sb * 128u;
                                for (int pass = 0; pass < passes; ++pass) {
    #pragma unroll
                                    for (int kk = 0; kk < kBN / 16; ++kk) {
                                        const uint64_t bd = sdesc_sw128(vb + kk * 16 * 128, kBN * 128, 1024);
                                        umma_bf16_ts(tmem + C::o_col(mt),
                                                     pa + (kk >> 2) * 64 + pass * 32 + (kk & 3) * 8, bd,
                                                     idesc_o, (first && pass == 0 && kk == 0) ? 0u : 1u);
                                    }
                                }
                                umma_commit(&ctrl->p_empty[sb]);
                                if (mt == NUM_MT - 1) {
                                    umma_commit(&ctrl->kv_empty[st]);
                                    if (cp.last()) umma_commit(&ctrl->o_full);
                                    CPA_TRACE_EVENT(14, gp);
                                    cp.advance(p, ctrl);
                                    if (++st_p == p.n_stages) {
                                        st_p = 0;
                                        par_p ^= 1u;
                                    }
                                }
                                ++ip;
                                progressed = true;
                            }
                        }
                    };
                    if (NUM_MT == 2) {
                        try_pv();
                        try_s();
                    } else {
                        try_s();
                        try_pv();
                    }
                    // Nothing ready: poll again.  (Suspending on the barrier that gates
                    // the next item, with a 0-200 ns hint or a 32-100 ns sleep, woke no
                    // sooner and cost the Llama-shaped call about 1 %.)
                    if (progressed) spins = 0;
                    if (!progressed && (++spins & 63u) == 0) {
                        // same time limit as every other wait of the kernel
                        const uint64_t now = globaltimer_ns();
                        if (spins == 64) t_idle = now;
                        if (*abort_flag) {
                            ok = false;
                        } else if (now - t_idle > kWaitLimitNs) {
                            atomicOr(p.status, CPA_DEV_TIMEOUT);
                            *abort_flag = 1u;
                            ok = false;
                        }
                        if (!ok) break;
                    }
                }
                umma_commit(&ctrl->mma_done);
                mbar_wait(&ctrl->mma_done, 0, abort_flag, p.status);
                CPA_TRACE_CTA(3, globaltimer_ns());
            }
            __syncwarp();
        } else if (FP8 && (warp == 2 || warp == 3)) {
            // ============================== FP8 widening (warps 2 and 3)
            // A stage's E4M3 K and V rows land in the hi-half regions (128 codes =
            // 128 B per row, 128-B swizzled like every operand row).  Each thread
            // widens whole rows in place, exactly: it reads a row's 128 codes, then
            // writes columns 0..63 as f16 to the lo-half region and columns 64..127
            // over the 128 B it read.  Thread ct owns rows ct and ct + 64 of K (the
            // S MMA waits for cv_full), then of V (the PV MMA waits for cvv_full).
            // V rows that hold no key of the sequence (not loaded, or past its end:
            // stale or arbitrary bytes, NaN codes included) are zeroed instead, so
            // that P = 0 takes them out exactly; stale K rows are masked columns.
            const int ct = (int)threadIdx.x - 64;
            int st = 0;
            uint32_t par = 0;
            const long long n_tiles = ctrl->count;
            for (long long g = 0; g < n_tiles; ++g) {
                uint8_t* stage = smem + p.off_kv + st * kStageBytes;
                bool okc = true;
#pragma unroll 1
                for (int kv = 0; kv < 2 && okc; ++kv) {
                    if (kv == 0) okc = mbar_wait_warp(&ctrl->kv_full[st], par, abort_flag, p.status);
                    if (!okc) break;
                    if (ct == 0 && kv == 0) CPA_TRACE_EVENT(57, g);
#pragma unroll 1
                    for (int i = 0; i < 2; ++i) {
                        const int r = ct + 64 * i, sw = r & 7;
                        uint8_t* lo = stage + (2 * kv) * (kBN * 128) + r * 128;
                        uint8_t* hi = lo + kBN * 128;
                        if (kv == 1 && !(ctrl->vrows[st][r >> 5] >> (r & 31) & 1u)) {
                            // (chunks in swizzled order, like every other access: the
                            // rows of 8 neighbouring lanes then fall in distinct banks)
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                *reinterpret_cast<uint4*>(lo + ((j ^ sw) << 4)) = make_uint4(0u, 0u, 0u, 0u);
                                *reinterpret_cast<uint4*>(hi + ((j ^ sw) << 4)) = make_uint4(0u, 0u, 0u, 0u);
                            }
                            continue;
                        }
                        uint4 c[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            c[j] = *reinterpret_cast<const uint4*>(hi + ((j ^ sw) << 4));
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            // codes 16j..16j+15 -> f16 columns 16j..16j+15: 16-B chunks
                            // 2(j%4) and 2(j%4)+1 of the lo (j < 4) or hi half
                            uint8_t* row = j < 4 ? lo : hi;
                            const int ca = 2 * (j & 3);
                            const uint4 a = make_uint4(e4m3x2_to_f16x2(c[j].x, false),
                                                       e4m3x2_to_f16x2(c[j].x, true),
                                                       e4m3x2_to_f16x2(c[j].y, false),
                                                       e4m3x2_to_f16x2(c[j].y, true));
                            const uint4 b = make_uint4(e4m3x2_to_f16x2(c[j].z, false),
                                                       e4m3x2_to_f16x2(c[j].z, true),
                                                       e4m3x2_to_f16x2(c[j].w, false),
                                                       e4m3x2_to_f16x2(c[j].w, true));
                            *reinterpret_cast<uint4*>(row + ((ca ^ sw) << 4)) = a;
                            *reinterpret_cast<uint4*>(row + (((ca + 1) ^ sw) << 4)) = b;
                        }
                    }
                    fence_proxy_async_smem();  // the tensor cores read these rows
                    __syncwarp();
                    if (lane == 0) mbar_arrive(kv == 0 ? &ctrl->cv_full[st] : &ctrl->cvv_full[st]);
                    if (ct == 0) CPA_TRACE_EVENT(kv == 0 ? 58 : 60, g);
                }
                if (!okc) break;
                if (++st == p.n_stages) {
                    st = 0;
                    par ^= 1u;
                }
            }
        } else if (warp >= C::kSmWarp0 && warp < C::kEpiWarp0) {
            // ============================== softmax
            // NUM_MT = 1: warpgroup `half` handles columns [64*half, 64*half + 64) of
            // every 128-key tile for all 128 rows; the two threads of a row swap
            // their partial maxima each tile so both apply the same running max.
            // NUM_MT = 2: warpgroup `mt` handles all 128 columns of its M tile.
            const int wgi = (warp - C::kSmWarp0) >> 2;
            const int mt = C::kSplit == 2 ? 0 : wgi;
            const int half = C::kSplit == 2 ? wgi : 0;
            const int quarter = warp & 3;
            const int r = quarter * 32 + lane;
            const int R = mt * 128 + r;
            const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
            const uint32_t o_addr = tmem + lane_addr + C::o_col(mt);
            constexpr int kChunks = 2 / C::kSplit;  // 64-column chunks per thread
            unsigned long long vis_keep = 0ull;  // tree, two M tiles: the masks of
            int vis_b = -1;                      // request vis_b's tree
            Walker w;
            w.init(ctrl);
            long long g = 0;
            bool ok = true;
            while (w.left > 0 && ok) {
                const Unit x = get_unit(p, w.u);
                int jb, je;
                w.piece(x, jb, je);
                const int it = R / G;
                int lo = x.lo, hi;
                if (is_verify(p.mode) || p.mode == MODE_PREFILL_RECT) hi = x.hi;
                else hi = p.H_hit + x.p0 + it + 1;
                // running max (log2 units, scaled) and this thread's part of the sum.
                // Rows past the unit's tokens are computed over whole tiles like the
                // others, so that a warp holding both kinds takes the unmasked path;
                // their results stay in their own O rows and are never written.
                float m_used = neg_inf(), l = 0.f;
                const bool warp_inert = __all_sync(0xffffffffu, it >= x.ntok);
                // keys [lo, hi_all) are visible to every row of this warp (rows past the
                // unit's tokens see whole prefix tiles): a prefix tile inside that range
                // is whole for the warp without the per-piece votes
                const int hi_all = __reduce_min_sync(0xffffffffu, it < x.ntok ? hi : INT_MAX);
                // tree verify: the tree tile's columns this row's node sees, its
                // ancestor-or-self mask (tutorial section 8.2: M[i, j] = 1 iff j is in
                // A(i)).  Every warp holds the request's parent array in registers
                // (lane l: parents l and l + 32) and each thread climbs its own node's
                // chain with warp shuffles (at most N steps, each to a smaller index;
                // an index outside [-1, i) stops the climb and sets CPA_DEV_BAD_TREE).
                // Warp-local, so no barrier across warps; done before a unit's first
                // tile.  With two M tiles the masks of the request's previous unit
                // (another KV head, the same tree) are kept: 221.2 -> 219.5 us on
                // 60-node trees; with one M tile keeping them live cost 1 us, so there
                // they are rebuilt for every unit.
                unsigned long long vis = NUM_MT == 2 ? vis_keep : 0ull;
                if (TREE && je == x.n_tiles && (NUM_MT == 1 || x.b != vis_b)) {
                    vis_b = x.b;
                    const int32_t* tpar = p.tree_par + (size_t)x.b * p.S;
                    const int tpar_lo = lane < p.S ? __ldg(tpar + lane) : -1;
                    const int tpar_hi = lane + 32 < p.S ? __ldg(tpar + lane + 32) : -1;
                    bool act = it < x.ntok;
                    int j = it;
                    vis = act ? 1ull << it : 0ull;
                    for (int step = 0; step < p.S; ++step) {
                        if (!__any_sync(0xffffffffu, act)) break;
                        const int a = __shfl_sync(0xffffffffu, tpar_lo, j & 31);
                        const int b = __shfl_sync(0xffffffffu, tpar_hi, j & 31);
                        const int pj = j < 32 ? a : b;
                        if (act) {
                            if (pj == -1) {
                                act = false;
                            } else if (pj < -1 || pj >= j) {
                                atomicOr(p.status, CPA_DEV_BAD_TREE);
                                act = false;
                            } else {
                                vis |= 1ull << pj;
                                j = pj;
                            }
                        }
                    }
                    if (NUM_MT == 2) vis_keep = vis;
                }
                for (int jj = jb; jj < je; ++jj, ++g) {
                    // this warpgroup's item: S buffer g % 2 (one M tile) or mt (two)
                    const int sb = (int)(g % C::kSBufs);
                    const int bi = C::kSBufs == 2 ? sb : mt;
                    const uint32_t par = (uint32_t)((C::kSBufs == 2 ? g >> 1 : g) & 1);
                    bool okl = mbar_wait_warp(&ctrl->s_full[bi], par, abort_flag, p.status);
                    if (threadIdx.x == C::kSmWarp0 * 32) CPA_TRACE_EVENT(4, g);
                    if (lane == 0) CPA_TRACE_EVENT(20 + warp - C::kSmWarp0, g);
                    const bool dtile = !PREFILL && jj >= x.n_prefix;
                    const bool tree_tile = TREE && dtile;
                    const int key0 = (x.tile_base + jj) * kBN;
                    // (not in the FP8 instance: it measured 5 % slower with it)
                    const bool tile_whole = !FP8 && !dtile && key0 >= lo && key0 + kBN <= hi_all;
                    // visible columns [lo_c, hi_c) of this tile for this row
                    int lo_c, hi_c;
                    if (dtile) {
                        // drafts: row (branch k, draft s) sees drafts 0..s of branch k,
                        // held in tile columns k*sb .. k*sb+s
                        const bool casc = p.mode == MODE_CASCADE;
                        lo_c = (casc ? it / p.S : 0) * p.sb;
                        hi_c = it < x.ntok ? lo_c + (casc ? it % p.S : it) + 1 : lo_c;
                    } else {
                        lo_c = lo - key0;
                        hi_c = hi - key0;
                    }
                    if (it >= x.ntok) {
                        lo_c = 0;
                        hi_c = dtile ? 0 : kBN;
                    }
                    const uint32_t s_addr = tmem + lane_addr + C::s_col(mt, sb);
                    if (okl) tc_fence_after_sync();
                    // Both passes walk this thread's columns in 32-column pieces.  A piece
                    // is, for the whole warp, unseen (no row sees any of it: not read, P = 0),
                    // whole (every row sees all of it) or partial (masked first).  Every tile
                    // runs the same per-piece code, so the rare masked tiles at a unit's end
                    // find it already in the instruction cache; only the masking is extra.
                    // (the tree tile: the columns of the row's ancestor mask)
                    auto tree_bits = [&](int a) -> uint32_t {
                        return a < 64 ? (uint32_t)(vis >> a) : 0u;
                    };
                    auto piece_class = [&](int a) -> int {  // 0 unseen, 1 partial, 2 whole
                        if (tree_tile) {
                            const uint32_t bits = tree_bits(a);
                            if (!__any_sync(0xffffffffu, bits != 0u)) return 0;
                            return __all_sync(0xffffffffu, bits == 0xffffffffu) ? 2 : 1;
                        }
                        if (!__any_sync(0xffffffffu, lo_c < a + 32 && hi_c > a)) return 0;
                        return __all_sync(0xffffffffu, lo_c <= a && hi_c >= a + 32) ? 2 : 1;
                    };
                    auto mask_piece = [&](uint32_t (&v)[32], int a) {
                        if (tree_tile) {
                            const uint32_t bits = tree_bits(a);
#pragma unroll
                            for (int c = 0; c < 32; ++c)
                                if (!(bits >> c & 1u)) v[c] = __float_as_uint(neg_inf());
                            return;
                        }
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            if (a + c < lo_c || a + c >= hi_c) v[c] = __float_as_uint(neg_inf());
                    };
                    // pass 1: this thread's raw maximum over its columns
                    float tmax_raw = neg_inf();
                    if (okl && !warp_inert) {
                        float m4[4] = {neg_inf(), neg_inf(), neg_inf(), neg_inf()};
#pragma unroll 1
                        for (int pc = 0; pc < 2 * kChunks; ++pc) {
                            const int a = half * 64 + (pc >> 1) * 64 * C::kSplit + (pc & 1) * 32;
                            const int cls = tile_whole ? 2 : piece_class(a);
                            if (cls == 0) continue;
                            uint32_t sv[32];
                            tmem_ld_x32(s_addr + (uint32_t)a, sv);
                            if (cls == 1) mask_piece(sv, a);
#pragma unroll
                            for (int c = 0; c < 8; ++c)
                                m4[c & 3] = fmax3(m4[c & 3], fmax3(__uint_as_float(sv[4 * c]),
                                                                   __uint_as_float(sv[4 * c + 1]),
                                                                   __uint_as_float(sv[4 * c + 2])),
                                                  __uint_as_float(sv[4 * c + 3]));
                        }
                        tmax_raw = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                    }
                    if (threadIdx.x == C::kSmWarp0 * 32) CPA_TRACE_EVENT(13, g);
                    if (lane == 0) CPA_TRACE_EVENT(28 + warp - C::kSmWarp0, g);
                    if (C::kSplit == 2) {
                        // swap partial maxima with the warp holding the other half of the
                        // same rows (a barrier of just that pair); it also makes the
                        // timeout decision common to both
                        xchg[((int)(g & 1) * 2 + half) * 128 + r] = tmax_raw;
                        okl = bar_and(4 + quarter, 64, okl);
                        tmax_raw = fmaxf(tmax_raw, xchg[((int)(g & 1) * 2 + (half ^ 1)) * 128 + r]);
                    }
                    if (!okl) {
                        ok = false;
                        break;
                    }
                    if (threadIdx.x == C::kSmWarp0 * 32) CPA_TRACE_EVENT(1, g);
                    if (lane == 0) CPA_TRACE_EVENT(36 + warp - C::kSmWarp0, g);
                    if (!warp_inert) {
                        const float tmax = tmax_raw * p.scale_log2;
                        const bool need = (m_used != neg_inf()) && (tmax > m_used + kRescaleLog2);
                        if (__any_sync(0xffffffffu, need)) {
                            // O holds PV of tiles up to g-1 of this unit: wait for it, then
                            // scale this thread's columns of O for rows whose max jumped
                            const int pb = C::kSBufs == 2 ? (int)((g - 1) & 1) : mt;
                            const uint32_t ppar =
                                (uint32_t)((C::kSBufs == 2 ? (g - 1) >> 1 : g - 1) & 1);
                            if (!mbar_wait_warp(&ctrl->p_empty[pb], ppar, abort_flag, p.status)) {
                                ok = false;  // the next barrier vote carries it to all threads
                            } else {
                                tc_fence_after_sync();
                                const float f = need ? ex2(m_used - tmax) : 1.f;
#pragma unroll 1
                                for (int c4 = 0; c4 < 4 / C::kSplit; ++c4) {
                                    const uint32_t oc = (uint32_t)(half * 64 + c4 * 32);
                                    uint32_t ov[32];
                                    tmem_ld_x32(o_addr + oc, ov);
#pragma unroll
                                    for (int i = 0; i < 32; ++i)
                                        ov[i] = __float_as_uint(__uint_as_float(ov[i]) * f);
                                    tmem_st_x32(o_addr + oc, ov);
                                }
                                if (need) {
                                    l *= f;
                                    m_used = tmax;
                                }
                            }
                        }
                        if (threadIdx.x == C::kSmWarp0 * 32) CPA_TRACE_EVENT(17, g);
                        if (m_used == neg_inf()) m_used = tmax;
                        const float mref = (m_used == neg_inf()) ? 0.f : m_used;
                        const bool resid = jj == x.resid_tile;
                        // pass 2: P = 2^(s*scale - mref) in bf16, written over the S columns
                        // it came from: piece k of a 64-column chunk puts its P in columns
                        // 16k..16k+15 of the chunk (S there is already read).  (The MMA that
                        // produced S is done, and so is every earlier MMA: no PV still reads
                        // these columns.)
                        // (scores scaled and the sum kept two at a time: one packed f32x2
                        // FMA and one packed add per pair of columns)
                        float2 s2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                        const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
                        const float2 nm2 = make_float2(-mref, -mref);
                        auto exp_piece = [&](const uint32_t (&sv)[32], uint32_t (&pk)[16]) {
#pragma unroll
                            for (int c = 0; c < 16; ++c) {
                                const float2 t = __ffma2_rn(make_float2(__uint_as_float(sv[2 * c]),
                                                                        __uint_as_float(sv[2 * c + 1])),
                                                            sc2, nm2);
                                const float ea = ex2(t.x), eb = ex2(t.y);
                                s2[c & 1] = __fadd2_rn(s2[c & 1], make_float2(ea, eb));
                                pk[c] = FP8 ? pack_f16x2(ea, eb) : pack_bf16x2(ea, eb);
                            }
                        };
                        if (FP8 || !resid) {
#pragma unroll 1
                            for (int pc = 0; pc < 2 * kChunks; ++pc) {
                                const int c0 = half * 64 + (pc >> 1) * 64 * C::kSplit;
                                const int a = c0 + 32 * (pc & 1);
                                const int cls = tile_whole ? 2 : piece_class(a);
                                uint32_t pk[16];
                                if (cls == 0) {
#pragma unroll
                                    for (int c = 0; c < 16; ++c) pk[c] = 0u;
                                } else {
                                    uint32_t sv[32];
                                    tmem_ld_x32(s_addr + (uint32_t)a, sv);
                                    if (cls == 1) mask_piece(sv, a);
                                    exp_piece(sv, pk);
                                }
                                tmem_st_x16_nowait(s_addr + (uint32_t)(c0 + 16 * (pc & 1)), pk);
                            }
                        } else {
                            // a small unit's last tile: the bf16 residual of P (what the
                            // rounding dropped) goes to columns 32.. of the chunk, which
                            // hold the second piece's S, so it is written once that piece
                            // has been read
#pragma unroll 1
                            for (int ch = 0; ch < kChunks; ++ch) {
                                const int c0 = (half + ch) * 64;
                                uint32_t rk0[16];
#pragma unroll 1
                                for (int sc = 0; sc < 2; ++sc) {
                                    const int a = c0 + 32 * sc;
                                    uint32_t pk[16], rk[16];
                                    if (!tile_whole && piece_class(a) == 0) {
#pragma unroll
                                        for (int c = 0; c < 16; ++c) pk[c] = rk[c] = 0u;
                                    } else {
                                        uint32_t sv[32];
                                        tmem_ld_x32(s_addr + (uint32_t)a, sv);
                                        mask_piece(sv, a);
                                        exp_piece(sv, pk);
#pragma unroll
                                        for (int c = 0; c < 16; ++c) {
                                            const float ea = ex2(
                                                fmaf(__uint_as_float(sv[2 * c]), p.scale_log2, -mref));
                                            const float eb = ex2(fmaf(__uint_as_float(sv[2 * c + 1]),
                                                                      p.scale_log2, -mref));
                                            rk[c] = pack_bf16x2(ea - __uint_as_float(pk[c] << 16),
                                                                eb - __uint_as_float(pk[c] & 0xFFFF0000u));
                                        }
                                    }
                                    tmem_st_x16_nowait(s_addr + (uint32_t)(c0 + 16 * sc), pk);
                                    if (sc == 0) {
#pragma unroll
                                        for (int c = 0; c < 16; ++c) rk0[c] = rk[c];
                                    } else {
                                        tmem_st_x16_nowait(s_addr + (uint32_t)(c0 + 32), rk0);
                                        tmem_st_x16_nowait(s_addr + (uint32_t)(c0 + 48), rk);
                                    }
                                }
                            }
                        }
                        tmem_wait_st();
                        l += (s2[0].x + s2[0].y) + (s2[1].x + s2[1].y);
                    }
                    if (threadIdx.x == C::kSmWarp0 * 32) CPA_TRACE_EVENT(5, g);
                    if (lane == 0) CPA_TRACE_EVENT(44 + warp - C::kSmWarp0, g);
                    bool zeroed = false;
                    // (FP8: the widening warps zero the V rows that hold no key)
                    const bool ztail = dtile ? (tree_tile && p.S % p.boxr != 0)
                                             : (key0 + kBN > x.valid_end && x.valid_end % p.boxr != 0);
                    if (!FP8 && wgi == 0 && ztail) {
                        // the box holding the sequence's last key (or the tree's last node)
                        // was loaded whole: zero its V rows past the end (whatever the page
                        // holds there), so that P = 0 contributes exactly nothing
                        const int first = tree_tile ? p.S : max(0, x.valid_end - key0);
                        const int stop = min(kBN, (first / p.boxr + 1) * p.boxr);
                        const int st = (int)(g % p.n_stages);
                        uint8_t* vb = smem + p.off_kv + st * kStageBytes + 2 * kBN * 128;
                        for (int i = r; i < 2 * (stop - first) * 8; i += 128) {
                            const int hh = i & 1, rem = i >> 1;  // rem: 16-B chunk within the rows
                            *reinterpret_cast<uint4*>(vb + hh * kBN * 128 + first * 128 + rem * 16) =
                                make_uint4(0, 0, 0, 0);
                        }
                        zeroed = true;
                    }
                    if (zeroed) fence_proxy_async_smem();  // the MMA reads those V rows
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ctrl->p_full[bi]);
                    if (threadIdx.x == C::kSmWarp0 * 32) CPA_TRACE_EVENT(6, g);
                    if (lane == 0 && wgi == 0) CPA_TRACE_EVENT(9 + quarter, g);
                }
                if (C::kSplit == 2) {
                    // the second half hands its part of each row sum to the first
                    if (half == 1) xsum[r] = l;
                    ok = bar_and(3, 256, ok);
                    if (half == 0) l += xsum[r];
                }
                if (!ok) break;
                if (half == 0) {
                    if (w.seg >= 1) {
                        ok = mbar_wait_warp(&ctrl->o_empty, (uint32_t)((w.seg - 1) & 1), abort_flag,
                                            p.status);
                    }
                    if (ok) {
                        stats[R] = make_float2(m_used, l);
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&ctrl->stats_full);
                    }
                }
                if (C::kSplit == 2) ok = bar_and(3, 256, ok);  // xsum and stats reuse
                w.next(x, jb, je, ctrl);
            }
        } else if (warp >= C::kEpiWarp0) {
            // ============================== epilogue
            // O / l for each row of a finished unit.  A unit split across CTAs is
            // written as a partial (o, lse); the CTA that completes it last merges
            // the partials in CTA order by the log-sum-exp identity.  With one M
            // tile, this warpgroup also loads each unit's Q rows into TMEM two
            // units ahead of use.
            const int quarter = warp & 3;
            const int r = quarter * 32 + lane;
            const int et = r;  // 0..127 within the epilogue warpgroup
            const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
            const bool fp32_out = p.out_f32 != 0;
            // Q of one unit into TMEM buffer qb: row r is query token r / G, head r % G.
            auto load_q = [&](const Unit& xu, int qb) {
                const int it = r / G, gq = r % G;
                const uint4* src = reinterpret_cast<const uint4*>(
                    p.q + ((size_t)(xu.t0 + (it < xu.ntok ? it : 0)) * p.H_q + xu.h * G + gq) * 128);
                if (FP8) {
                    // FP8 pools: q * k_scale (the unit's KV head) in f16, 32 columns
                    // (64 channels) at a time
                    const float* ks = p.k_scale + (p.scale_per_channel ? xu.h * 128 : 0);
                    const int cs = p.scale_per_channel ? 1 : 0;
#pragma unroll 1
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t v[32];
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            uint4 u = make_uint4(0u, 0u, 0u, 0u);
                            if (it < xu.ntok) u = __ldg(src + hh * 8 + c);
                            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const int ch = (hh * 8 + c) * 8 + 2 * k;  // channel of the low half
                                v[4 * c + k] = pack_f16x2(__uint_as_float(w[k] << 16) * __ldg(ks + cs * ch),
                                                          __uint_as_float(w[k] & 0xFFFF0000u) *
                                                              __ldg(ks + cs * (ch + 1)));
                            }
                        }
                        __syncwarp();
                        tmem_st_x32(tmem + lane_addr + C::q_col(qb) + 32u * hh, v);
                    }
                } else {
                    uint32_t v[64];
                    if (it < xu.ntok) {
                        uint4 u[16];
#pragma unroll
                        for (int c = 0; c < 16; ++c) u[c] = __ldg(src + c);
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            v[4 * c] = u[c].x;
                            v[4 * c + 1] = u[c].y;
                            v[4 * c + 2] = u[c].z;
                            v[4 * c + 3] = u[c].w;
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < 64; ++c) v[c] = 0u;
                    }
                    __syncwarp();
                    tmem_st_x64(tmem + lane_addr + C::q_col(qb), v);
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctrl->q_full[qb]);
            };
            Walker wq;  // runs two units ahead of `w` to stage Q
            wq.init(ctrl);
            int q_loaded = 0;
            if (C::kQInTmem) {
                for (; q_loaded < 2 && wq.left > 0; ++q_loaded) {
                    const Unit xq = get_unit(p, wq.u);
                    int qjb, qje;
                    wq.piece(xq, qjb, qje);
                    load_q(xq, q_loaded);
                    wq.next(xq, qjb, qje, ctrl);
                }
            }
            Walker w;
            w.init(ctrl);
            bool ok = true;
            while (w.left > 0 && ok) {
                const Unit x = get_unit(p, w.u);
                int jb, je;
                w.piece(x, jb, je);
                const bool split = !PREFILL && (jb > 0 || je < x.n_tiles);
                const uint32_t ph = (uint32_t)(w.seg & 1);
                ok = mbar_wait(&ctrl->o_full, ph, abort_flag, p.status) &&
                     mbar_wait(&ctrl->stats_full, ph, abort_flag, p.status);
                ok = bar_and(1, 128, ok);  // one decision for the whole epilogue warpgroup
                if (!ok) break;
                if (et == 0) CPA_TRACE_EVENT(7, w.seg);
                tc_fence_after_sync();

                // Write one row; oa(blk, f) supplies columns blk*32..+31 of its output.
                auto finish_row = [&](int R, float lse2, auto&& oa) {
                    const int it = R / G, gq = R % G;
                    const bool valid = it < x.ntok;
                    const size_t orow = (size_t)(x.t0 + (valid ? it : 0)) * p.H_q + x.h * G + gq;
                    // weights of the merge with another level's part (p.mrg_o), log2 units
                    float mw_own = 1.f, mw_oth = 0.f;
                    if (MERGE && valid) {
                        const float lm = __ldg(p.mrg_lse + orow);
                        const float lo = lm == neg_inf() ? neg_inf() : lm * kLog2e;
                        if (lse2 == neg_inf() && lo == neg_inf()) {
                            mw_own = 0.f;
                        } else {
                            const float mx = fmaxf(lse2, lo);
                            const float a = ex2(lse2 - mx), b = ex2(lo - mx);
                            mw_own = a / (a + b);
                            mw_oth = b / (a + b);
                            lse2 = mx + lg2(a + b);
                        }
                    }
#pragma unroll 1
                    for (int blk = 0; blk < 4; ++blk) {
                        float f[32];
                        __syncwarp();
                        oa(blk, f);
                        if (!valid) continue;
                        if (MERGE) {
                            // merge with the other level's part of this row:
                            // o = 2^(lse2 - lm) o_own + 2^(lo - lm) o_other
#pragma unroll
                            for (int e = 0; e < 32; ++e) f[e] *= mw_own;
                            const float4* src =
                                reinterpret_cast<const float4*>(p.mrg_o + orow * 128 + blk * 32);
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const float4 v = __ldg(src + e);
                                f[4 * e] = fmaf(mw_oth, v.x, f[4 * e]);
                                f[4 * e + 1] = fmaf(mw_oth, v.y, f[4 * e + 1]);
                                f[4 * e + 2] = fmaf(mw_oth, v.z, f[4 * e + 2]);
                                f[4 * e + 3] = fmaf(mw_oth, v.w, f[4 * e + 3]);
                            }
                        }
                        if (FP8) {
                            // the V scale, per tensor or per (KV head, channel)
                            const float* vs =
                                p.v_scale + (p.scale_per_channel ? x.h * 128 + blk * 32 : 0);
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                f[e] *= __ldg(vs + (p.scale_per_channel ? e : 0));
                        }
                        if (fp32_out) {
                            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) +
                                                                    orow * 128 + blk * 32);
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                dst[e] = make_float4(f[4 * e], f[4 * e + 1], f[4 * e + 2],
                                                     f[4 * e + 3]);
                        } else {
                            uint4* dst = reinterpret_cast<uint4*>(
                                static_cast<__nv_bfloat16*>(p.o) + orow * 128 + blk * 32);
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                dst[e] = make_uint4(pack_bf16x2(f[8 * e], f[8 * e + 1]),
                                                    pack_bf16x2(f[8 * e + 2], f[8 * e + 3]),
                                                    pack_bf16x2(f[8 * e + 4], f[8 * e + 5]),
                                                    pack_bf16x2(f[8 * e + 6], f[8 * e + 7]));
                        }
                    }
                    if (valid) p.lse[orow] = lse2 == neg_inf() ? neg_inf() : lse2 * kLn2;
                };

                if (!split) {
                    for (int mt = 0; mt < NUM_MT; ++mt) {
                        const int R = mt * 128 + r;
                        const float2 st = stats[R];
                        const float lse2 = st.y > 0.f ? st.x + lg2(st.y) : neg_inf();
                        const float inv = st.y > 0.f ? 1.f / st.y : 0.f;
                        const uint32_t oaddr = tmem + lane_addr + C::o_col(mt);
                        finish_row(R, lse2, [&](int blk, float (&f)[32]) {
                            uint32_t v[32];
                            tmem_ld_x32(oaddr + blk * 32, v);
#pragma unroll
                            for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(v[e]) * inv;
                        });
                    }
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ctrl->o_empty);
                } else {
                    // A unit split over CTAs c_first..c_last: the piece that finishes last
                    // merges all pieces, in CTA order, so the result does not depend on
                    // which one that is.  A piece that finds every other piece already
                    // stored is that last one and takes its own part straight from TMEM;
                    // otherwise it stores its part (O / l and its log-sum-exp) and counts
                    // itself in, and the piece that completes the count merges.
                    const int c_first = split_owner(total, n_ctas, w.ustart, kFast32);
                    const int c_last = split_owner(total, n_ctas, w.ustart + x.n_tiles - 1, kFast32);
                    const int np = c_last - c_first + 1;
                    const int own = (int)blockIdx.x - c_first;
                    // (only as the CTA's final piece: a merge holds O in TMEM, and any
                    // later unit of this CTA waits for it)
                    const bool final_piece = w.left == (long long)(je - jb);
                    if (et == 0) {
                        const unsigned seen = final_piece ? ld_acquire_gpu(p.counters + w.u) : 0u;
                        ctrl->flag = (final_piece && seen == (unsigned)(np - 1)) ? 2 : 0;
                    }
                    named_bar_sync(1, 128);
                    int mode = *reinterpret_cast<volatile int*>(&ctrl->flag);
                    if (mode == 0) {
                        // the part stays in L2 until the merging CTA reads it, typically
                        // at the very end, after the whole K/V stream has passed through
                        const uint64_t pol_keep = l2_policy_evict_last();
                        const int slot = split_slot(total, n_ctas, blockIdx.x, w.ustart, kFast32);
                        for (int mt = 0; mt < NUM_MT; ++mt) {
                            const int R = mt * 128 + r;
                            const float2 st = stats[R];
                            const float lse2 = st.y > 0.f ? st.x + lg2(st.y) : neg_inf();
                            const float inv = st.y > 0.f ? 1.f / st.y : 0.f;
                            const uint32_t oaddr = tmem + lane_addr + C::o_col(mt);
                            const bool valid = R / G < x.ntok;
                            // float4 group q of every row side by side: a warp's store
                            // of one group covers 512 contiguous bytes
                            float4* po = reinterpret_cast<float4*>(p.part_o) +
                                         (size_t)slot * 32 * kMaxUnitRows + R;
#pragma unroll 1
                            for (int blk = 0; blk < 4; ++blk) {
                                uint32_t v[32];
                                __syncwarp();
                                tmem_ld_x32(oaddr + blk * 32, v);
                                if (valid) {
#pragma unroll
                                    for (int e = 0; e < 8; ++e)
                                        st_global_hint(po + (blk * 8 + e) * kPartRows,
                                                       make_float4(__uint_as_float(v[4 * e]) * inv,
                                                                   __uint_as_float(v[4 * e + 1]) * inv,
                                                                   __uint_as_float(v[4 * e + 2]) * inv,
                                                                   __uint_as_float(v[4 * e + 3]) * inv),
                                                       pol_keep);
                                }
                            }
                            if (valid) p.part_lse[(size_t)slot * kMaxUnitRows + R] = lse2;
                        }
                        if (et == 0) CPA_TRACE_EVENT(52, w.seg);
                        tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&ctrl->o_empty);
                        __threadfence();
                        named_bar_sync(1, 128);
                        if (et == 0) CPA_TRACE_EVENT(53, w.seg);
                        if (et == 0) {
                            const unsigned old = atomicAdd(p.counters + w.u, 1u);
                            ctrl->flag = (old == (unsigned)(np - 1)) ? 1 : 0;
                        }
                        named_bar_sync(1, 128);
                        mode = *reinterpret_cast<volatile int*>(&ctrl->flag);
                        if (et == 0) CPA_TRACE_EVENT(54, w.seg);
                    }
                    if (mode != 0) {
                        // mode 2: this piece's part comes from TMEM, the others' from memory.
                        // As the CTA's final piece every K/V stage is idle (all MMAs are
                        // done): each other part is bulk-copied there whole (one copy of
                        // its contiguous slot), so that the merge waits on memory once.
                        // (mode 1 counted itself in with a relaxed atomic: fence before
                        // reading the others' parts; mode 2 read the count with acquire)
                        if (mode == 1) __threadfence();
                        const int nl = kPartRows;  // log-sum-exp entries copied per part
                        const uint32_t part_bytes = 32u * (uint32_t)kPartRows * 16u;
                        const uint32_t lse_off = (uint32_t)(np - 1) * part_bytes;
                        const bool staged = mode == 2 && lse_off + (uint32_t)(np - 1) * nl * 4u <=
                                                             (uint32_t)p.n_stages * kStageBytes;
                        const float4* stage4 = reinterpret_cast<const float4*>(smem + p.off_kv);
                        const float* stage_lse = reinterpret_cast<const float*>(smem + p.off_kv + lse_off);
                        if (staged) {
                            if (et < 32) {
                                // lane k of the first epilogue warp copies the k-th other part
                                // and its log-sum-exp entries
                                fence_proxy_async_global();
                                if (et == 0)
                                    mbar_arrive_expect_tx(&ctrl->merge_full,
                                                          lse_off + (uint32_t)(np - 1) * nl * 4u);
                                __syncwarp();
                                const int k = et;
                                if (k < np - 1) {
                                    const int c = k < own ? k : k + 1;
                                    const size_t sl =
                                        split_slot(total, n_ctas, c_first + c, w.ustart, kFast32);
                                    bulk_load(smem + p.off_kv + (size_t)k * part_bytes,
                                              reinterpret_cast<const float4*>(p.part_o) +
                                                  sl * 32 * kMaxUnitRows,
                                              part_bytes, &ctrl->merge_full);
                                    bulk_load(smem + p.off_kv + lse_off + (size_t)k * nl * 4,
                                              p.part_lse + sl * kMaxUnitRows, (uint32_t)nl * 4u,
                                              &ctrl->merge_full);
                                }
                            }
                            // at most one staged merge per CTA: phase 0
                            const bool okm = bar_and(1, 128, mbar_wait(&ctrl->merge_full, 0,
                                                                       abort_flag, p.status));
                            if (!okm) {
                                ok = false;
                                break;
                            }
                        }
                        if (et == 0) CPA_TRACE_EVENT(55, w.seg);
                        for (int mt = 0; mt < NUM_MT; ++mt) {
                            const int R = mt * 128 + r;
                            const bool valid = R / G < x.ntok;
                            const float2 st = stats[R];
                            const float lse_own = st.y > 0.f ? st.x + lg2(st.y) : neg_inf();
                            const float inv = st.y > 0.f ? 1.f / st.y : 0.f;
                            const uint32_t oaddr = tmem + lane_addr + C::o_col(mt);
                            auto slot_of = [&](int c) -> size_t {
                                return (size_t)split_slot(total, n_ctas, c_first + c, w.ustart, kFast32);
                            };
                            auto lse_of = [&](int c) -> float {
                                if (mode == 2 && c == own) return lse_own;
                                if (staged) return stage_lse[(c < own ? c : c - 1) * nl + R];
                                return __ldcg(p.part_lse + slot_of(c) * kMaxUnitRows + R);
                            };
                            // log2 of the sum of 2^lse over the parts, as a running (max, sum)
                            float mx = neg_inf(), den = 0.f;
                            if (valid) {
#pragma unroll 4
                                for (int c = 0; c < np; ++c) {
                                    const float lc = lse_of(c);
                                    if (lc == neg_inf()) continue;
                                    if (lc > mx) {
                                        den = (mx == neg_inf() ? 0.f : den * ex2(mx - lc)) + 1.f;
                                        mx = lc;
                                    } else {
                                        den += ex2(lc - mx);
                                    }
                                }
                            }
                            const float lse2 = (den > 0.f) ? mx + lg2(den) : neg_inf();
                            if (et == 0) CPA_TRACE_EVENT(56, w.seg);
                            finish_row(R, lse2, [&](int blk, float (&f)[32]) {
                                uint32_t v[32];
                                if (mode == 2) tmem_ld_x32(oaddr + blk * 32, v);
#pragma unroll
                                for (int e = 0; e < 32; ++e) f[e] = 0.f;
                                if (!valid || den == 0.f) return;
                                for (int c = 0; c < np; ++c) {
                                    const float wc = ex2(lse_of(c) - lse2);
                                    if (mode == 2 && c == own) {
#pragma unroll
                                        for (int e = 0; e < 32; ++e)
                                            f[e] = fmaf(wc, __uint_as_float(v[e]) * inv, f[e]);
                                        continue;
                                    }
                                    float4 v4[8];
                                    if (staged) {
                                        const float4* s4 =
                                            stage4 + ((size_t)(c < own ? c : c - 1) * 32 + blk * 8) * kPartRows + R;
#pragma unroll
                                        for (int e = 0; e < 8; ++e) v4[e] = s4[e * kPartRows];
                                    } else {
                                        const float4* s4 = reinterpret_cast<const float4*>(p.part_o) +
                                                           slot_of(c) * 32 * kMaxUnitRows +
                                                           (size_t)blk * 8 * kPartRows + R;
#pragma unroll
                                        for (int e = 0; e < 8; ++e) v4[e] = __ldcg(s4 + e * kPartRows);
                                    }
#pragma unroll
                                    for (int e = 0; e < 8; ++e) {
                                        f[4 * e] = fmaf(wc, v4[e].x, f[4 * e]);
                                        f[4 * e + 1] = fmaf(wc, v4[e].y, f[4 * e + 1]);
                                        f[4 * e + 2] = fmaf(wc, v4[e].z, f[4 * e + 2]);
                                        f[4 * e + 3] = fmaf(wc, v4[e].w, f[4 * e + 3]);
                                    }
                                }
                            });
                        }
                        if (mode == 2) {
                            tc_fence_before_sync();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&ctrl->o_empty);
                        }
                    }
                }
                if (et == 0) CPA_TRACE_EVENT(8, w.seg);
                // Q of the unit two ahead goes into the buffer this unit used: every
                // MMA of this unit is done (o_full), so nothing reads it any more
                if (C::kQInTmem && wq.left > 0) {
                    const Unit xq = get_unit(p, wq.u);
                    int qjb, qje;
                    wq.piece(xq, qjb, qje);
                    load_q(xq, q_loaded % 2);
                    ++q_loaded;
                    wq.next(xq, qjb, qje, ctrl);
                }
                w.next(x, jb, je, ctrl);
            }
            if (et == 0) {
                CPA_TRACE_CTA(4, globaltimer_ns());
                CPA_TRACE_CTA(6, (unsigned long long)w.seg);
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
#ifdef CPA_TRACE
    if (threadIdx.x == 0 && cpa_trace_local) {
        if (blockIdx.x < 4) {
            cpa_trace_local[(blockIdx.x * 64 + kTraceStampRow) * 1024 + 2] = clock64();
            cpa_trace_local[(blockIdx.x * 64 + kTraceStampRow) * 1024 + 3] = globaltimer_ns();
        }
        CPA_TRACE_CTA(1, globaltimer_ns());
    }
#endif
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

}  // namespace cpa
