// cpa_api.cu -- the extern "C" entry points of libcpa.so: argument checks,
// TMA tensor maps, workspace layout and kernel launches.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "cpa.h"
#include "cpa_attn.cuh"
#include "cpa_host.h"
#include "cpa_small.h"

namespace cpa {
namespace {

constexpr size_t kStatusBytes = 256;
constexpr int kMaxSmemOptin = 232448;  // 227 KB per CTA on sm_100-class parts

// ---------------------------------------------------------------- device facts
int smem_optin() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return 0;
    return n;
}

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

// ---------------------------------------------------------------- tensor maps
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// bf16 tensor [dim2][dim1][128] seen as (d, dim1, dim2), 128-B swizzled boxes
// of {64, box1, box2}.
bool make_map(CUtensorMap* map, const void* base, uint64_t dim1, uint64_t dim2, uint32_t box1,
              uint32_t box2) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {128, dim1, dim2};
    cuuint64_t strides[2] = {128 * 2, dim1 * 128 * 2};
    cuuint32_t box[3] = {64, box1, box2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// uint8 tensor (FP8 E4M3 codes) [dim2][dim1][128] seen as (d, dim1, dim2),
// 128-B swizzled boxes of {128, box1, box2}: one box row is a whole 128-code row.
bool make_map_u8(CUtensorMap* map, const void* base, uint64_t dim1, uint64_t dim2,
                 uint32_t box1, uint32_t box2) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {128, dim1, dim2};
    cuuint64_t strides[2] = {128, dim1 * 128};
    cuuint32_t box[3] = {128, box1, box2};
    cuuint32_t estr[3] = {1, 1, 1};
    // 128-B L2 promotion: a row of one head is 128 B here, and 256-B promotion
    // (right for bf16, whose 256-B rows are fetched as two halves) would fetch
    // the neighbouring head's row with every row
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }
bool page_size_ok(int P) { return P >= 8 && P <= 256 && pow2(P); }
size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ---------------------------------------------------------------- workspace layout
struct WsLayout {
    size_t counters, part_lse, part_o, total;
};
WsLayout ws_layout(long long n_units, int n_sm) {
    WsLayout w;
    w.counters = kStatusBytes;
    w.part_lse = align_up(w.counters + (size_t)n_units * 4, 256);
    w.part_o = align_up(w.part_lse + (size_t)2 * n_sm * kMaxUnitRows * 4, 256);
    w.total = align_up(w.part_o + (size_t)2 * n_sm * kMaxUnitRows * 128 * 4, 256);
    return w;
}

// Tree verify: the fused kernel's workspace (the kernel builds the ancestor
// masks itself, from the parent array).
size_t tree_ws_bytes(int B, int H_kv, int n_sm) {
    return ws_layout((long long)B * H_kv, n_sm).total;
}

// Multi-level verify: the larger of the two launches' workspaces, then the
// shared level's fp32 partial (the own level merges it into its output).
struct SharedWs {
    size_t attn, o1, lse1, total;
};
SharedWs shared_ws_layout(int B, int n_groups, int topk, int S, int H_q, int H_kv, int n_sm) {
    SharedWs w;
    const int G = H_q / H_kv;
    const int TS = 128 / G;
    const long long M = (long long)(B / n_groups) * topk * S;
    const long long QT = (M + TS - 1) / TS;
    const size_t a1 = ws_layout((long long)n_groups * H_kv * QT, n_sm).total;
    const size_t a2 = ws_layout((long long)B * H_kv, n_sm).total;
    const size_t rows = (size_t)B * topk * S * H_q;
    w.attn = a1 > a2 ? a1 : a2;
    w.o1 = w.attn;
    w.lse1 = align_up(w.o1 + rows * 128 * 4, 256);
    w.total = align_up(w.lse1 + rows * 4, 256);
    return w;
}

// ---------------------------------------------------------------- launch config
struct Geometry {
    int num_mt;
    int TS, TSB, Rq;
    int n_stages, n_qbufs;
    uint32_t off_q, off_kv;
    int smem_bytes;
};

// Shared-memory plan: control block, row statistics and exchange buffers,
// then (units of two M tiles only) the Q tile, then the K/V stage ring with
// as many 64 KB stages as fit (up to 4).  Units of one M tile keep Q in
// tensor memory, double-buffered.
bool plan_geometry(int G, int TS, Geometry& g) {
    const int rows = TS * G;
    if (rows <= 0 || rows > kMaxUnitRows) return false;
    g.num_mt = rows <= 128 ? 1 : 2;
    g.TS = TS;
    g.TSB = g.num_mt == 1 ? TS : 128 / G;
    const int rows_mt = G * g.TSB;
    if (rows_mt > 128) return false;
    g.Rq = (rows_mt + 7) / 8 * 8;
    const size_t qmt = (size_t)2 * g.Rq * 128;
    g.n_qbufs = g.num_mt == 1 ? 2 : 1;
    const size_t off_q = kOffData;
    const size_t q_bytes = g.num_mt == 1 ? 0 : (size_t)g.num_mt * qmt;
    const size_t off_kv = align_up(off_q + q_bytes, 1024);
    for (int st = 4; st >= 2; --st) {
        const size_t total = off_kv + (size_t)st * kStageBytes + 1024;
        if (total <= (size_t)kMaxSmemOptin) {
            g.n_stages = st;
            g.off_q = (uint32_t)off_q;
            g.off_kv = (uint32_t)off_kv;
            g.smem_bytes = (int)total;
            return true;
        }
    }
    return false;
}

// The dynamic shared-memory limit of a kernel is an attribute of the device's
// context, so it is raised once per device (and per kernel instance), not once
// per process: a process that drives several GPUs from one library instance
// needs it on each of them.
template <int NUM_MT, int VAR>
cudaError_t raise_smem_limit_once() {
    static PerDevice<int> state;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    return (cudaError_t)state.run(dev, (int)cudaErrorInvalidDevice, [](int&) {
        const int optin = smem_optin();
        return (int)cudaFuncSetAttribute(paged_attn_kernel<NUM_MT, VAR>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         optin < kMaxSmemOptin ? optin : kMaxSmemOptin);
    });
}

template <int NUM_MT, int VAR>
cudaError_t launch_attn(const AttnParams& p, int smem, int grid, cudaStream_t stream) {
    cudaError_t e = raise_smem_limit_once<NUM_MT, VAR>();
    if (e != cudaSuccess) return e;
    if (smem > smem_optin()) return cudaErrorInvalidValue;
    paged_attn_kernel<NUM_MT, VAR><<<grid, Cfg<NUM_MT>::kThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

template <int VAR>
cudaError_t launch_attn_mt(const AttnParams& p, const Geometry& geo, int grid,
                           cudaStream_t stream) {
    return geo.num_mt == 1 ? launch_attn<1, VAR>(p, geo.smem_bytes, grid, stream)
                           : launch_attn<2, VAR>(p, geo.smem_bytes, grid, stream);
}

// keep_status: the call is the second launch of one entry point, whose first
// launch already cleared the status word (clearing it again would drop that
// launch's bits); only the merge counters are cleared.
cpa_status run_attn(AttnParams& p, const Geometry& geo, long long n_units, void* workspace,
                    size_t ws_bytes, cudaStream_t stream, bool keep_status = false) {
    const int n_sm = sm_count();
    if (n_sm <= 0) return CPA_ERR_CUDA;
    const WsLayout wl = ws_layout(n_units, n_sm);
    if (!workspace) return CPA_ERR_WORKSPACE;
    if (ws_bytes < wl.total) return CPA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return CPA_ERR_INVALID_ARG;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    p.status = reinterpret_cast<uint32_t*>(ws);
    p.counters = reinterpret_cast<uint32_t*>(ws + wl.counters);
    p.part_lse = reinterpret_cast<float*>(ws + wl.part_lse);
    p.part_o = reinterpret_cast<float*>(ws + wl.part_o);
    p.TS = geo.TS;
    p.TSB = geo.TSB;
    p.Rq = geo.Rq;
    p.n_stages = geo.n_stages;
    p.n_qbufs = geo.n_qbufs;
    p.off_q = geo.off_q;
    p.off_kv = geo.off_kv;
    const size_t clear0 = keep_status ? wl.counters : 0;
    if (cudaMemsetAsync(ws + clear0, 0, wl.part_lse - clear0, stream) != cudaSuccess)
        return CPA_ERR_CUDA;
    // the FP8 instance exists for one M tile only (Q is staged in TMEM as f16)
    if (p.fp8 && geo.num_mt != 1) return CPA_ERR_UNSUPPORTED;
    cudaError_t e;
    if (p.fp8)
        e = launch_attn<1, VAR_FP8>(p, geo.smem_bytes, n_sm, stream);
    else if (p.mode == MODE_TREE)
        e = launch_attn_mt<VAR_TREE>(p, geo, n_sm, stream);
    else if (p.mrg_o)
        e = launch_attn_mt<VAR_MERGE>(p, geo, n_sm, stream);
    else if ((p.mode == MODE_PREFILL || p.mode == MODE_PREFILL_TRI) && geo.num_mt == 1)
        e = launch_attn<1, VAR_PREFILL>(p, geo.smem_bytes, n_sm, stream);
    else
        e = launch_attn_mt<VAR_PLAIN>(p, geo, n_sm, stream);
    return e == cudaSuccess ? CPA_OK : CPA_ERR_LAUNCH;
}

// Checks shared by the verify entry points.
cpa_status check_verify(const void* q, const void* k_pages, const void* v_pages,
                        const int32_t* ppt, int ppt_stride, const int32_t* lens, int B, int topk,
                        int S, int H_q, int H_kv, int head_dim, int page_size, int num_pages,
                        int max_prefix_len, float sm_scale) {
    if (!q || !k_pages || !v_pages || !ppt || !lens) return CPA_ERR_INVALID_ARG;
    if (B < 1 || topk < 1 || S < 1 || H_q < 1 || H_kv < 1 || num_pages < 1 || max_prefix_len < 0)
        return CPA_ERR_INVALID_ARG;
    if (H_q % H_kv != 0) return CPA_ERR_INVALID_ARG;
    if (!(sm_scale > 0.f) || !std::isfinite(sm_scale)) return CPA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages)) return CPA_ERR_INVALID_ARG;
    if (head_dim != 128) return CPA_ERR_UNSUPPORTED;
    if (!page_size_ok(page_size)) return CPA_ERR_UNSUPPORTED;
    const int G = H_q / H_kv;
    if (!pow2(G) || G > 128) return CPA_ERR_UNSUPPORTED;
    const long long need_pages = ((long long)max_prefix_len + page_size - 1) / page_size;
    if (ppt_stride < 1 || ppt_stride < need_pages) return CPA_ERR_INVALID_ARG;
    if ((long long)num_pages * page_size > (1ll << 31)) return CPA_ERR_UNSUPPORTED;
    if ((long long)B * topk * S * H_q > (1ll << 31) / 128) return CPA_ERR_UNSUPPORTED;
    return CPA_OK;
}

void fill_common(AttnParams& p, const void* q, const void* k_pages, const void* v_pages,
                 const int32_t* ppt, int ppt_stride, const int32_t* dpt, int dpt_stride,
                 const int32_t* lens, int B, int topk, int S, int H_q, int H_kv, int page_size,
                 int num_pages, int max_prefix_len, float sm_scale) {
    std::memset(&p, 0, sizeof p);
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.k_pages = static_cast<const __nv_bfloat16*>(k_pages);
    p.v_pages = static_cast<const __nv_bfloat16*>(v_pages);
    p.ptab = ppt;
    p.ptab_stride = ppt_stride;
    p.dtab = dpt;
    p.dtab_stride = dpt_stride;
    p.lens = lens;
    p.B = B;
    p.topk = topk;
    p.S = S;
    p.H_q = H_q;
    p.H_kv = H_kv;
    p.G = H_q / H_kv;
    p.P = page_size;
    p.num_pages = num_pages;
    p.max_len = max_prefix_len;
    p.s_grp = 1;
    p.boxr = page_size < kBN ? page_size : kBN;
    p.scale_log2 = sm_scale * kLog2e;
}

// K/V pool maps with `rows`-row boxes: bf16 pools in 64-column halves, FP8
// pools in whole 128-code rows.
bool pool_map(const AttnParams& p, CUtensorMap* map, const void* base, int H_kv,
              uint64_t pool_rows, uint32_t rows) {
    return p.fp8 ? make_map_u8(map, base, H_kv, pool_rows, 1, rows)
                 : make_map(map, base, H_kv, pool_rows, 1, rows);
}

bool kv_maps(AttnParams& p, const void* k_pages, const void* v_pages, int H_kv, int num_pages,
             int page_size) {
    const uint64_t rows = (uint64_t)num_pages * page_size;
    return pool_map(p, &p.kmap, k_pages, H_kv, rows, p.boxr) &&
           pool_map(p, &p.vmap, v_pages, H_kv, rows, p.boxr);
}

// Scales of FP8 E4M3 pools: one K and one V value, or [H_kv, 128] each.
struct Fp8Scales {
    const float* k_scale;
    const float* v_scale;
    int per_channel;
};

// f32_out: o receives the fp32 result (always for Pass A; for cascade when the
// result is a partial that a later launch merges).  keep_status: see run_attn.
// A prefix segment shared by groups of `grp` consecutive requests: `len`
// logical positions (whole pages) read through row b / grp of `table`, before
// each request's own prefix.
struct SharedSeg {
    const int32_t* table;
    int stride, len, grp;
};

// fp8: the pools hold E4M3 codes with these scales (one M tile only).
// Tree verify (MODE_TREE): dpt is the tree table, S the node count N (topk 1)
// and tree_par the parent array [B][N].
cpa_status verify_common(int mode, const void* q, const void* k_pages, const void* v_pages,
                         const int32_t* ppt, int ppt_stride, const int32_t* dpt, int dpt_stride,
                         const int32_t* lens, int B, int topk, int S, int H_q, int H_kv,
                         int head_dim, int page_size, int num_pages, int max_prefix_len,
                         float sm_scale, void* o, float* lse, void* workspace, size_t ws_bytes,
                         cudaStream_t stream, bool f32_out = false, bool keep_status = false,
                         const Fp8Scales* fp8 = nullptr,
                         const int32_t* tree_par = nullptr,
                         const float* mrg_o = nullptr, const float* mrg_lse = nullptr,
                         const SharedSeg* seg = nullptr) {
    cpa_status st = check_verify(q, k_pages, v_pages, ppt, ppt_stride, lens, B, topk, S, H_q, H_kv,
                                 head_dim, page_size, num_pages, max_prefix_len, sm_scale);
    if (st != CPA_OK) return st;
    if (!o || !lse || !aligned16(o)) return CPA_ERR_INVALID_ARG;
    if (fp8 && (!fp8->k_scale || !fp8->v_scale ||
                (reinterpret_cast<uintptr_t>(fp8->k_scale) & 3u) ||
                (reinterpret_cast<uintptr_t>(fp8->v_scale) & 3u)))
        return CPA_ERR_INVALID_ARG;
    const bool draft = mode != MODE_PASS_A;
    const bool tree = mode == MODE_TREE;
    // The draft tile holds each branch's drafts in a block of sb rows, all read
    // from the branch's first draft page (tree verify: the tree's nodes in rows
    // 0..S-1, read through the tree table).
    const int sb = S <= 8 ? 8 : 16;
    const int nbr = mode == MODE_CASCADE ? topk : 1;
    if (draft) {
        if (!dpt || dpt_stride < (S + page_size - 1) / page_size) return CPA_ERR_INVALID_ARG;
        if (tree ? (S > CPA_MAX_TREE_NODES || !tree_par || fp8)
                 : (S > kMaxDraft || S > page_size || nbr * sb > kBN))
            return CPA_ERR_UNSUPPORTED;
    }
    const int G = H_q / H_kv;
    const int TS = mode == MODE_NAIVE ? S : topk * S;
    Geometry geo;
    if (!plan_geometry(G, TS, geo)) return CPA_ERR_UNSUPPORTED;
    if (fp8 && geo.num_mt != 1) return CPA_ERR_UNSUPPORTED;
    AttnParams p;
    fill_common(p, q, k_pages, v_pages, ppt, ppt_stride, dpt, dpt_stride, lens, B, topk, S, H_q,
                H_kv, page_size, num_pages, max_prefix_len, sm_scale);
    if (fp8) {
        p.fp8 = 1;
        p.k_scale = fp8->k_scale;
        p.v_scale = fp8->v_scale;
        p.scale_per_channel = fp8->per_channel ? 1 : 0;
    }
    p.mode = mode;
    p.out_f32 = (mode == MODE_PASS_A || f32_out) ? 1 : 0;
    p.upg = mode == MODE_NAIVE ? topk * H_kv : H_kv;
    p.has_draft = draft ? 1 : 0;
    p.sb = sb;
    p.nbr = nbr;
    p.tree_par = tree_par;
    if (seg) {
        p.stab = seg->table;
        p.stab_stride = seg->stride;
        p.s_len = seg->len;
        p.s_grp = seg->grp;
    }
    p.mrg_o = mrg_o;
    p.mrg_lse = mrg_lse;
    p.o = o;
    p.lse = lse;
    const uint64_t T = (uint64_t)B * topk * S;
    if (!make_map(&p.qmap, q, H_q, T, G, geo.TSB)) return CPA_ERR_CUDA;
    if (!kv_maps(p, k_pages, v_pages, H_kv, num_pages, page_size)) return CPA_ERR_CUDA;
    if (draft && !tree) {
        const uint64_t rows = (uint64_t)num_pages * page_size;
        // a branch's draft box is exactly its S rows: the rest of the branch block
        // keeps earlier, finite tile data, which P = 0 there multiplies away
        if (!pool_map(p, &p.kdmap, k_pages, H_kv, rows, S) ||
            !pool_map(p, &p.vdmap, v_pages, H_kv, rows, S))
            return CPA_ERR_CUDA;
    }
    const long long n_units = (long long)B * p.upg;
    return run_attn(p, geo, n_units, workspace, ws_bytes, stream, keep_status);
}

}  // namespace
}  // namespace cpa

using namespace cpa;

extern "C" {

const char* cpa_status_string(cpa_status s) {
    switch (s) {
        case CPA_OK: return "ok";
        case CPA_ERR_INVALID_ARG: return "invalid argument";
        case CPA_ERR_UNSUPPORTED: return "unsupported configuration";
        case CPA_ERR_WORKSPACE: return "workspace missing or too small";
        case CPA_ERR_LAUNCH: return "kernel launch failed";
        case CPA_ERR_BAD_PAGE: return "page id out of range";
        case CPA_ERR_TIMEOUT: return "device wait timed out";
        case CPA_ERR_CUDA: return "CUDA runtime error";
        case CPA_ERR_BAD_LENGTH: return "prefix length out of range";
        case CPA_ERR_BAD_TREE: return "tree parent index out of range";
    }
    return "unknown status";
}

int cpa_version(void) { return 100; }

size_t cpa_status_workspace_size(void) { return kStatusBytes; }

size_t cpa_cascade_verify_workspace_size(int B, int topk, int S, int H_q, int H_kv, int head_dim,
                                         int page_size) {
    if (B < 1 || topk < 1 || S < 1 || H_q < 1 || H_kv < 1 || H_q % H_kv || head_dim != 128 ||
        !page_size_ok(page_size))
        return 0;
    const int n_sm = sm_count();
    if (n_sm <= 0) return 0;
    return ws_layout((long long)B * topk * H_kv, n_sm).total;
}

cpa_status cpa_cascade_verify(const void* q, const void* k_pages, const void* v_pages,
                              const int32_t* prefix_page_table, int prefix_pt_stride,
                              const int32_t* draft_page_table, int draft_pt_stride,
                              const int32_t* prefix_lens, int B, int topk, int S, int H_q,
                              int H_kv, int head_dim, int page_size, int num_pages,
                              int max_prefix_len, float sm_scale, void* o, float* lse,
                              void* workspace, size_t workspace_bytes, cpa_stream_t stream) {
    return verify_common(MODE_CASCADE, q, k_pages, v_pages, prefix_page_table, prefix_pt_stride,
                         draft_page_table, draft_pt_stride, prefix_lens, B, topk, S, H_q, H_kv,
                         head_dim, page_size, num_pages, max_prefix_len, sm_scale, o, lse,
                         workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

cpa_status cpa_naive_expand_verify(const void* q, const void* k_pages, const void* v_pages,
                                   const int32_t* prefix_page_table, int prefix_pt_stride,
                                   const int32_t* draft_page_table, int draft_pt_stride,
                                   const int32_t* prefix_lens, int B, int topk, int S, int H_q,
                                   int H_kv, int head_dim, int page_size, int num_pages,
                                   int max_prefix_len, float sm_scale, void* o, float* lse,
                                   void* workspace, size_t workspace_bytes, cpa_stream_t stream) {
    return verify_common(MODE_NAIVE, q, k_pages, v_pages, prefix_page_table, prefix_pt_stride,
                         draft_page_table, draft_pt_stride, prefix_lens, B, topk, S, H_q, H_kv,
                         head_dim, page_size, num_pages, max_prefix_len, sm_scale, o, lse,
                         workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

cpa_status cpa_cascade_verify_fp8(const void* q, const void* k_pages, const void* v_pages,
                                  const float* k_scale, const float* v_scale,
                                  int scale_per_channel, const int32_t* prefix_page_table,
                                  int prefix_pt_stride, const int32_t* draft_page_table,
                                  int draft_pt_stride, const int32_t* prefix_lens, int B, int topk,
                                  int S, int H_q, int H_kv, int head_dim, int page_size,
                                  int num_pages, int max_prefix_len, float sm_scale, void* o,
                                  float* lse, void* workspace, size_t workspace_bytes,
                                  cpa_stream_t stream) {
    const Fp8Scales sc{k_scale, v_scale, scale_per_channel};
    return verify_common(MODE_CASCADE, q, k_pages, v_pages, prefix_page_table, prefix_pt_stride,
                         draft_page_table, draft_pt_stride, prefix_lens, B, topk, S, H_q, H_kv,
                         head_dim, page_size, num_pages, max_prefix_len, sm_scale, o, lse,
                         workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream),
                         false, false, &sc);
}

cpa_status cpa_cascade_pass_a_fp8(const void* q, const void* k_pages, const void* v_pages,
                                  const float* k_scale, const float* v_scale,
                                  int scale_per_channel, const int32_t* prefix_page_table,
                                  int prefix_pt_stride, const int32_t* prefix_lens, int B,
                                  int topk, int S, int H_q, int H_kv, int head_dim, int page_size,
                                  int num_pages, int max_prefix_len, float sm_scale, float* o_a,
                                  float* lse_a, void* workspace, size_t workspace_bytes,
                                  cpa_stream_t stream) {
    const Fp8Scales sc{k_scale, v_scale, scale_per_channel};
    return verify_common(MODE_PASS_A, q, k_pages, v_pages, prefix_page_table, prefix_pt_stride,
                         nullptr, 0, prefix_lens, B, topk, S, H_q, H_kv, head_dim, page_size,
                         num_pages, max_prefix_len, sm_scale, o_a, lse_a, workspace,
                         workspace_bytes, reinterpret_cast<cudaStream_t>(stream), false, false,
                         &sc);
}

cpa_status cpa_cascade_pass_a(const void* q, const void* k_pages, const void* v_pages,
                              const int32_t* prefix_page_table, int prefix_pt_stride,
                              const int32_t* prefix_lens, int B, int topk, int S, int H_q,
                              int H_kv, int head_dim, int page_size, int num_pages,
                              int max_prefix_len, float sm_scale, float* o_a, float* lse_a,
                              void* workspace, size_t workspace_bytes, cpa_stream_t stream) {
    return verify_common(MODE_PASS_A, q, k_pages, v_pages, prefix_page_table, prefix_pt_stride,
                         nullptr, 0, prefix_lens, B, topk, S, H_q, H_kv, head_dim, page_size,
                         num_pages, max_prefix_len, sm_scale, o_a, lse_a, workspace,
                         workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

cpa_status cpa_cascade_pass_b(const void* q, const void* k_pages, const void* v_pages,
                              const int32_t* draft_page_table, int draft_pt_stride, int B,
                              int topk, int S, int H_q, int H_kv, int head_dim, int page_size,
                              int num_pages, float sm_scale, float* o_b, float* lse_b,
                              void* workspace, size_t workspace_bytes, cpa_stream_t stream) {
    if (!q || !k_pages || !v_pages || !draft_page_table || !o_b || !lse_b)
        return CPA_ERR_INVALID_ARG;
    if (B < 1 || topk < 1 || S < 1 || H_q < 1 || H_kv < 1 || H_q % H_kv || num_pages < 1 ||
        page_size < 1 || !std::isfinite(sm_scale))
        return CPA_ERR_INVALID_ARG;
    if (head_dim != 128) return CPA_ERR_UNSUPPORTED;
    if (draft_pt_stride < (S + page_size - 1) / page_size) return CPA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(q) & 7u) || (reinterpret_cast<uintptr_t>(k_pages) & 7u) ||
        (reinterpret_cast<uintptr_t>(v_pages) & 7u) || !aligned16(o_b))
        return CPA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < kStatusBytes) return CPA_ERR_WORKSPACE;
    PassBParams p;
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.k_pages = static_cast<const __nv_bfloat16*>(k_pages);
    p.v_pages = static_cast<const __nv_bfloat16*>(v_pages);
    p.dtab = draft_page_table;
    p.dtab_stride = draft_pt_stride;
    p.B = B;
    p.topk = topk;
    p.S = S;
    p.H_q = H_q;
    p.H_kv = H_kv;
    p.P = page_size;
    p.num_pages = num_pages;
    p.scale_log2 = sm_scale * kLog2e;
    p.o_b = o_b;
    p.lse_b = lse_b;
    p.status = static_cast<uint32_t*>(workspace);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(workspace, 0, kStatusBytes, s) != cudaSuccess) return CPA_ERR_CUDA;
    return launch_pass_b(p, s) == cudaSuccess ? CPA_OK : CPA_ERR_LAUNCH;
}

cpa_status cpa_merge_state(const float* o_a, const float* lse_a, const float* o_b,
                           const float* lse_b, int n_tokens, int H, int head_dim, void* o_out,
                           float* lse_out, cpa_stream_t stream) {
    if (!o_a || !lse_a || !o_b || !lse_b || !o_out || !lse_out) return CPA_ERR_INVALID_ARG;
    if (n_tokens < 0 || H < 1 || head_dim < 4 || head_dim % 4 != 0) return CPA_ERR_INVALID_ARG;
    if (head_dim > 512) return CPA_ERR_UNSUPPORTED;
    if (!aligned16(o_a) || !aligned16(o_b) || (reinterpret_cast<uintptr_t>(o_out) & 7u))
        return CPA_ERR_INVALID_ARG;
    const long long rows = (long long)n_tokens * H;
    if (rows == 0) return CPA_OK;
    const int n_sm = sm_count();
    if (n_sm <= 0) return CPA_ERR_CUDA;
    return launch_merge_state(o_a, lse_a, o_b, lse_b, rows, head_dim, o_out, lse_out, n_sm,
                              reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? CPA_OK
               : CPA_ERR_LAUNCH;
}

size_t cpa_prefill_hit_workspace_size(int B, int N, int H_hit, int H_q, int H_kv, int head_dim,
                                      int page_size) {
    if (B < 1 || N < 1 || H_hit < 0 || H_hit > N || H_q < 1 || H_kv < 1 || H_q % H_kv ||
        head_dim != 128 || !page_size_ok(page_size))
        return 0;
    const int G = H_q / H_kv;
    if (!pow2(G) || G > 128) return 0;
    const int n_sm = sm_count();
    if (n_sm <= 0) return 0;
    const int TS = 128 / G;
    const long long QT = ((long long)(N - H_hit) + TS - 1) / TS;
    return ws_layout((long long)B * H_kv * (QT > 0 ? QT : 1), n_sm).total;
}

cpa_status cpa_prefill_hit(const void* q, const void* k_pages, const void* v_pages,
                           const int32_t* page_table, int pt_stride, int B, int N, int H_hit,
                           int H_q, int H_kv, int head_dim, int page_size, int num_pages,
                           float sm_scale, int part, void* o, float* lse, void* workspace,
                           size_t workspace_bytes, cpa_stream_t stream) {
    if (!q || !k_pages || !v_pages || !page_table || !o || !lse) return CPA_ERR_INVALID_ARG;
    if (B < 1 || N < 1 || H_hit < 0 || H_hit > N || H_q < 1 || H_kv < 1 || H_q % H_kv ||
        num_pages < 1 || !(sm_scale > 0.f) || !std::isfinite(sm_scale))
        return CPA_ERR_INVALID_ARG;
    if (part != CPA_PREFILL_FULL && part != CPA_PREFILL_RECT && part != CPA_PREFILL_TRI)
        return CPA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(o))
        return CPA_ERR_INVALID_ARG;
    if (head_dim != 128 || !page_size_ok(page_size)) return CPA_ERR_UNSUPPORTED;
    const int G = H_q / H_kv;
    if (!pow2(G) || G > 128) return CPA_ERR_UNSUPPORTED;
    if (pt_stride < (N + page_size - 1) / page_size) return CPA_ERR_INVALID_ARG;
    if ((long long)num_pages * page_size > (1ll << 31)) return CPA_ERR_UNSUPPORTED;
    const int M = N - H_hit;
    if (M == 0) return CPA_OK;
    const int TS = 128 / G;
    Geometry geo;
    if (!plan_geometry(G, TS, geo)) return CPA_ERR_UNSUPPORTED;
    AttnParams p;
    fill_common(p, q, k_pages, v_pages, page_table, pt_stride, nullptr, 0, nullptr, B, 1, 1, H_q,
                H_kv, page_size, num_pages, 0, sm_scale);
    p.mode = part == CPA_PREFILL_FULL ? MODE_PREFILL
             : part == CPA_PREFILL_RECT ? MODE_PREFILL_RECT
                                        : MODE_PREFILL_TRI;
    p.out_f32 = part != CPA_PREFILL_FULL ? 1 : 0;
    p.N = N;
    p.H_hit = H_hit;
    p.M = M;
    p.QT = (M + TS - 1) / TS;
    p.o = o;
    p.lse = lse;
    if (!make_map(&p.qmap, q, H_q, (uint64_t)B * M, G, geo.TSB)) return CPA_ERR_CUDA;
    if (!kv_maps(p, k_pages, v_pages, H_kv, num_pages, page_size)) return CPA_ERR_CUDA;
    const long long n_units = (long long)B * H_kv * p.QT;
    return run_attn(p, geo, n_units, workspace, workspace_bytes,
                    reinterpret_cast<cudaStream_t>(stream));
}

size_t cpa_cascade_verify_shared_workspace_size(int B, int n_groups, int topk, int S, int H_q,
                                                int H_kv, int head_dim, int page_size) {
    if (B < 1 || n_groups < 1 || B % n_groups || topk < 1 || S < 1 || H_q < 1 || H_kv < 1 ||
        H_q % H_kv || head_dim != 128 || !page_size_ok(page_size))
        return 0;
    if (!pow2(H_q / H_kv) || H_q / H_kv > 128) return 0;
    const int n_sm = sm_count();
    if (n_sm <= 0) return 0;
    return shared_ws_layout(B, n_groups, topk, S, H_q, H_kv, n_sm).total;
}

cpa_status cpa_cascade_verify_shared(const void* q, const void* k_pages, const void* v_pages,
                                     const int32_t* shared_page_table, int shared_pt_stride,
                                     int n_groups, int shared_len,
                                     const int32_t* prefix_page_table, int prefix_pt_stride,
                                     const int32_t* draft_page_table, int draft_pt_stride,
                                     const int32_t* prefix_lens, int B, int topk, int S, int H_q,
                                     int H_kv, int head_dim, int page_size, int num_pages,
                                     int max_prefix_len, float sm_scale, void* o, float* lse,
                                     void* workspace, size_t workspace_bytes,
                                     cpa_stream_t stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // everything checkable is checked before the first launch
    cpa_status st = check_verify(q, k_pages, v_pages, prefix_page_table, prefix_pt_stride,
                                 prefix_lens, B, topk, S, H_q, H_kv, head_dim, page_size,
                                 num_pages, max_prefix_len, sm_scale);
    if (st != CPA_OK) return st;
    if (!o || !lse || !aligned16(o) || n_groups < 1 || B % n_groups || shared_len < 0)
        return CPA_ERR_INVALID_ARG;
    if (shared_len == 0)  // one level less: plain cascade verify
        return verify_common(MODE_CASCADE, q, k_pages, v_pages, prefix_page_table,
                             prefix_pt_stride, draft_page_table, draft_pt_stride, prefix_lens, B,
                             topk, S, H_q, H_kv, head_dim, page_size, num_pages, max_prefix_len,
                             sm_scale, o, lse, workspace, workspace_bytes, s);
    if (!shared_page_table || shared_pt_stride < (shared_len + page_size - 1) / page_size)
        return CPA_ERR_INVALID_ARG;
    const int sb = S <= 8 ? 8 : 16;
    if (!draft_page_table || draft_pt_stride < (S + page_size - 1) / page_size)
        return CPA_ERR_INVALID_ARG;
    if (S > kMaxDraft || S > page_size || topk * sb > kBN) return CPA_ERR_UNSUPPORTED;
    if (shared_len % page_size == 0) {
        // A whole number of shared pages: one launch.  Every (request, KV head)
        // unit walks its group's shared pages, then its own, then its drafts;
        // the requests of a group read the shared pages at about the same time,
        // so DRAM delivers them once and L2 serves the rest.  The kernel is
        // bound by per-tile work rather than by bytes, and this schedule has
        // the tiles of a single-level call, without the first level's short
        // units, its fp32 partial and a second launch.
        const SharedSeg seg{shared_page_table, shared_pt_stride, shared_len, B / n_groups};
        return verify_common(MODE_CASCADE, q, k_pages, v_pages, prefix_page_table,
                             prefix_pt_stride, draft_page_table, draft_pt_stride, prefix_lens, B,
                             topk, S, H_q, H_kv, head_dim, page_size, num_pages, max_prefix_len,
                             sm_scale, o, lse, workspace, workspace_bytes, s, false, false,
                             nullptr, nullptr, nullptr, nullptr, &seg);
    }
    // Otherwise two launches (the shared prefix ends inside a page).
    const int G = H_q / H_kv;
    Geometry geo1, geo2;
    if (!plan_geometry(G, 128 / G, geo1) || !plan_geometry(G, topk * S, geo2))
        return CPA_ERR_UNSUPPORTED;
    const int n_sm = sm_count();
    if (n_sm <= 0) return CPA_ERR_CUDA;
    const SharedWs w = shared_ws_layout(B, n_groups, topk, S, H_q, H_kv, n_sm);
    if (!workspace || workspace_bytes < w.total) return CPA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return CPA_ERR_INVALID_ARG;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    float* o1 = reinterpret_cast<float*>(ws + w.o1);
    float* lse1 = reinterpret_cast<float*>(ws + w.lse1);

    // level 1: the group's draft queries (consecutive tokens) against its shared
    // prefix, read once per group: the rectangle of a prefix-hit prefill whose
    // M suffix queries are the group's tokens and whose sequence ends with the
    // shared prefix (so no key past it is loaded)
    const int M = (B / n_groups) * topk * S;
    const int TS = 128 / G;
    AttnParams p;
    fill_common(p, q, k_pages, v_pages, shared_page_table, shared_pt_stride, nullptr, 0, nullptr,
                n_groups, 1, 1, H_q, H_kv, page_size, num_pages, 0, sm_scale);
    p.mode = MODE_PREFILL_RECT;
    p.out_f32 = 1;
    p.N = shared_len;
    p.H_hit = shared_len;
    p.M = M;
    p.QT = (M + TS - 1) / TS;
    p.o = o1;
    p.lse = lse1;
    if (!make_map(&p.qmap, q, H_q, (uint64_t)n_groups * M, G, geo1.TSB)) return CPA_ERR_CUDA;
    if (!kv_maps(p, k_pages, v_pages, H_kv, num_pages, page_size)) return CPA_ERR_CUDA;
    st = run_attn(p, geo1, (long long)n_groups * H_kv * p.QT, workspace, w.attn, s);
    if (st != CPA_OK) return st;
    // level 2: own prefix + drafts, the fused cascade kernel, which merges each
    // finished row with level 1's part of it (the LSE identity) and writes bf16 o
    return verify_common(MODE_CASCADE, q, k_pages, v_pages, prefix_page_table, prefix_pt_stride,
                         draft_page_table, draft_pt_stride, prefix_lens, B, topk, S, H_q, H_kv,
                         head_dim, page_size, num_pages, max_prefix_len, sm_scale, o, lse,
                         workspace, w.attn, s, /*f32_out=*/false, /*keep_status=*/true, nullptr,
                         nullptr, o1, lse1);
}

size_t cpa_tree_verify_workspace_size(int B, int N, int H_q, int H_kv, int head_dim,
                                      int page_size) {
    if (B < 1 || N < 1 || N > CPA_MAX_TREE_NODES || H_q < 1 || H_kv < 1 || H_q % H_kv ||
        head_dim != 128 || !page_size_ok(page_size))
        return 0;
    const int n_sm = sm_count();
    if (n_sm <= 0) return 0;
    return tree_ws_bytes(B, H_kv, n_sm);
}

cpa_status cpa_tree_verify(const void* q, const void* k_pages, const void* v_pages,
                           const int32_t* prefix_page_table, int prefix_pt_stride,
                           const int32_t* tree_page_table, int tree_pt_stride,
                           const int32_t* prefix_lens, const int32_t* tree_parents, int B, int N,
                           int H_q, int H_kv, int head_dim, int page_size, int num_pages,
                           int max_prefix_len, float sm_scale, void* o, float* lse,
                           void* workspace, size_t workspace_bytes, cpa_stream_t stream) {
    // everything checkable is checked before the launch
    cpa_status st = check_verify(q, k_pages, v_pages, prefix_page_table, prefix_pt_stride,
                                 prefix_lens, B, 1, N, H_q, H_kv, head_dim, page_size, num_pages,
                                 max_prefix_len, sm_scale);
    if (st != CPA_OK) return st;
    if (!tree_page_table || !tree_parents || !o || !lse || !aligned16(o))
        return CPA_ERR_INVALID_ARG;
    if (N > CPA_MAX_TREE_NODES) return CPA_ERR_UNSUPPORTED;
    if (tree_pt_stride < (N + page_size - 1) / page_size) return CPA_ERR_INVALID_ARG;
    Geometry geo;
    if (!plan_geometry(H_q / H_kv, N, geo)) return CPA_ERR_UNSUPPORTED;
    const int n_sm = sm_count();
    if (n_sm <= 0) return CPA_ERR_CUDA;
    if (!workspace || workspace_bytes < tree_ws_bytes(B, H_kv, n_sm)) return CPA_ERR_WORKSPACE;
    // one launch: the prefix once per request for all N nodes and the tree as one
    // more tile of the same online softmax, masked per row by the node's ancestor
    // mask (built in the kernel from the parent array), merged there
    return verify_common(MODE_TREE, q, k_pages, v_pages, prefix_page_table, prefix_pt_stride,
                         tree_page_table, tree_pt_stride, prefix_lens, B, 1, N, H_q, H_kv,
                         head_dim, page_size, num_pages, max_prefix_len, sm_scale, o, lse,
                         workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream),
                         /*f32_out=*/false, /*keep_status=*/false, nullptr, tree_parents);
}

cpa_status cpa_tree_pass_b(const void* q, const void* k_pages, const void* v_pages,
                           const int32_t* tree_page_table, int tree_pt_stride,
                           const int32_t* tree_parents, int B, int N, int H_q, int H_kv,
                           int head_dim, int page_size, int num_pages, float sm_scale,
                           float* o_b, float* lse_b, void* workspace, size_t workspace_bytes,
                           cpa_stream_t stream) {
    if (!q || !k_pages || !v_pages || !tree_page_table || !tree_parents || !o_b || !lse_b)
        return CPA_ERR_INVALID_ARG;
    if (B < 1 || N < 1 || H_q < 1 || H_kv < 1 || H_q % H_kv || num_pages < 1 || page_size < 1 ||
        !(sm_scale > 0.f) || !std::isfinite(sm_scale))
        return CPA_ERR_INVALID_ARG;
    if (head_dim != 128 || N > CPA_MAX_TREE_NODES) return CPA_ERR_UNSUPPORTED;
    if (tree_pt_stride < (N + page_size - 1) / page_size) return CPA_ERR_INVALID_ARG;
    if ((long long)B * N * H_q > (1ll << 31) / 128) return CPA_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(q) & 7u) || !aligned16(k_pages) || !aligned16(v_pages) ||
        !aligned16(o_b))
        return CPA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < kStatusBytes) return CPA_ERR_WORKSPACE;
    TreeParams tp;
    tp.q = static_cast<const __nv_bfloat16*>(q);
    tp.k_pages = static_cast<const __nv_bfloat16*>(k_pages);
    tp.v_pages = static_cast<const __nv_bfloat16*>(v_pages);
    tp.ttab = tree_page_table;
    tp.ttab_stride = tree_pt_stride;
    tp.parents = tree_parents;
    tp.B = B;
    tp.N = N;
    tp.H_q = H_q;
    tp.H_kv = H_kv;
    tp.P = page_size;
    tp.num_pages = num_pages;
    tp.scale_log2 = sm_scale * kLog2e;
    tp.o_a = nullptr;
    tp.lse_a = nullptr;
    tp.o = o_b;
    tp.lse = lse_b;
    tp.status = static_cast<uint32_t*>(workspace);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(workspace, 0, kStatusBytes, s) != cudaSuccess) return CPA_ERR_CUDA;
    return launch_tree(tp, s) == cudaSuccess ? CPA_OK : CPA_ERR_LAUNCH;
}

cpa_status cpa_get_device_status(const void* workspace, uint32_t* status_out,
                                  cpa_stream_t stream) {
    if (!workspace || !status_out) return CPA_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t v = 0;
    if (cudaMemcpyAsync(&v, workspace, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return CPA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return CPA_ERR_CUDA;
    *status_out = v;
    if (v & CPA_DEV_TIMEOUT) return CPA_ERR_TIMEOUT;
    if (v & CPA_DEV_BAD_PAGE) return CPA_ERR_BAD_PAGE;
    if (v & CPA_DEV_BAD_LENGTH) return CPA_ERR_BAD_LENGTH;
    if (v & CPA_DEV_BAD_TREE) return CPA_ERR_BAD_TREE;
    return CPA_OK;
}

cpa_status cpa_debug_wait_timeout(void* workspace, size_t workspace_bytes, int limit_us,
                                  cpa_stream_t stream) {
    if (!workspace || workspace_bytes < kStatusBytes) return CPA_ERR_WORKSPACE;
    if (limit_us < 1 || limit_us > 1000000) return CPA_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(workspace, 0, kStatusBytes, s) != cudaSuccess) return CPA_ERR_CUDA;
    return launch_wait_timeout(static_cast<uint32_t*>(workspace),
                               (unsigned long long)limit_us * 1000ull, s) == cudaSuccess
               ? CPA_OK
               : CPA_ERR_LAUNCH;
}

#ifdef CPA_TRACE
// Diagnostic builds only (compiled with -DCPA_TRACE; not part of the product
// library or its header): point the attention kernel's trace hooks at a
// caller-owned device buffer laid out as described in cpa_attn.cuh, or at
// nothing (NULL).  Returns 0 on success.
int cpa_trace_set_buffer(void* device_buffer) {
    return cudaMemcpyToSymbol(cpa_trace_buf, &device_buffer, sizeof device_buffer) == cudaSuccess
               ? 0
               : 1;
}
#endif

int cpa_plan_partition(int64_t total, int n_ctas, int cta, int64_t tile, int64_t* begin,
                       int64_t* end) {
    if (total < 1 || n_ctas < 1 || n_ctas > total || cta < 0 || cta >= n_ctas || tile < 0 ||
        tile >= total)
        return -1;
    const int64_t b = split_begin(total, n_ctas, cta), e = split_begin(total, n_ctas, cta + 1);
    const int owner = split_owner(total, n_ctas, tile);
    // the 32-bit form some kernel instances use must agree with the 64-bit one
    if (b != split_begin(total, n_ctas, cta, true) || e != split_begin(total, n_ctas, cta + 1, true) ||
        owner != split_owner(total, n_ctas, tile, true))
        return -2;
    if (begin) *begin = b;
    if (end) *end = e;
    return owner;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Static-scratch variant: the workspace is a file-scope device array, so this
// path allocates nothing.  Host code never passes g_static_scratch itself (in
// host code the name stands for a host-side shadow); it resolves the device
// address once per device with cudaGetSymbolAddress.
namespace {

static __device__ __align__(256) unsigned char g_static_scratch[CPA_STATIC_SCRATCH_BYTES];

PerDevice<void*> g_scratch_addr;

// Device address of this device's copy of the array (looked up on first use).
cpa_status static_scratch_for_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return CPA_ERR_CUDA;
    const int e = g_scratch_addr.run(dev, (int)CPA_ERR_CUDA, [](void*& p) {
        return cudaGetSymbolAddress(&p, g_static_scratch) == cudaSuccess ? 0 : (int)CPA_ERR_CUDA;
    }, out);
    return (cpa_status)e;
}

}  // namespace

extern "C" {

cpa_status cpa_cascade_verify_noalloc(const void* q, const void* k_pages, const void* v_pages,
                                      const int32_t* prefix_page_table, int prefix_pt_stride,
                                      const int32_t* draft_page_table, int draft_pt_stride,
                                      const int32_t* prefix_lens, int B, int topk, int S, int H_q,
                                      int H_kv, int head_dim, int page_size, int num_pages,
                                      int max_prefix_len, float sm_scale, void* o, float* lse,
                                      cpa_stream_t stream) {
    // the argument checks of the workspace call come first, so a bad size is
    // reported as such and not as a scratch shortage
    cpa_status st = check_verify(q, k_pages, v_pages, prefix_page_table, prefix_pt_stride,
                                 prefix_lens, B, topk, S, H_q, H_kv, head_dim, page_size,
                                 num_pages, max_prefix_len, sm_scale);
    if (st != CPA_OK) return st;
    const int n_sm = sm_count();
    if (n_sm <= 0) return CPA_ERR_CUDA;
    // the cascade launch has one work unit per (request, KV head)
    if (ws_layout((long long)B * H_kv, n_sm).total > (size_t)CPA_STATIC_SCRATCH_BYTES)
        return CPA_ERR_WORKSPACE;
    void* scratch = nullptr;
    st = static_scratch_for_current_device(&scratch);
    if (st != CPA_OK) return st;
    return verify_common(MODE_CASCADE, q, k_pages, v_pages, prefix_page_table, prefix_pt_stride,
                         draft_page_table, draft_pt_stride, prefix_lens, B, topk, S, H_q, H_kv,
                         head_dim, page_size, num_pages, max_prefix_len, sm_scale, o, lse,
                         scratch, (size_t)CPA_STATIC_SCRATCH_BYTES,
                         reinterpret_cast<cudaStream_t>(stream));
}

cpa_status cpa_noalloc_device_status(uint32_t* status_out, cpa_stream_t stream) {
    if (!status_out) return CPA_ERR_INVALID_ARG;
    void* scratch = nullptr;
    const cpa_status st = static_scratch_for_current_device(&scratch);
    if (st != CPA_OK) return st;
    return cpa_get_device_status(scratch, status_out, stream);
}

}  // extern "C"
