// cpa_small.cu -- the light kernels of the library: merge_state, the
// stand-alone Pass B draft kernel, the draft-tree pass, and the bounded-wait
// check.
#include <cuda_runtime.h>

#include "cpa_device.cuh"
#include "cpa_small.h"

namespace cpa {

namespace {
constexpr float kLog2eF = 1.4426950408889634f;
constexpr float kLn2F = 0.6931471805599453f;

__device__ __forceinline__ float ninf() { return __int_as_float(0xff800000); }
}  // namespace

// merge_state ("Cascade attention" page, split property):
//   lse = log(e^a + e^b), o = e^(a-lse) o_a + e^(b-lse) o_b,
// evaluated about m = max(a, b).  One thread per 4 consecutive elements of a
// row; consecutive threads cover consecutive addresses (16-B loads, 8-B stores).
__global__ void __launch_bounds__(256) merge_state_kernel(const float* __restrict__ o_a,
                                                          const float* __restrict__ lse_a,
                                                          const float* __restrict__ o_b,
                                                          const float* __restrict__ lse_b,
                                                          long long n_rows, int d4,
                                                          __nv_bfloat16* __restrict__ o_out,
                                                          float* __restrict__ lse_out) {
    const long long n = n_rows * d4;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        const long long row = i / d4;
        const int c4 = (int)(i - row * d4);
        const float a = __ldg(lse_a + row), b = __ldg(lse_b + row);
        float wa, wb, lse;
        if (a == ninf() && b == ninf()) {
            wa = 0.f;
            wb = 0.f;
            lse = ninf();
        } else {
            const float m = fmaxf(a, b);
            const float ea = ex2((a - m) * kLog2eF), eb = ex2((b - m) * kLog2eF);
            const float s = ea + eb;
            wa = ea / s;
            wb = eb / s;
            lse = m + lg2(s) * kLn2F;
        }
        const float4 x = __ldg(reinterpret_cast<const float4*>(o_a) + i);
        const float4 y = __ldg(reinterpret_cast<const float4*>(o_b) + i);
        const uint2 out = make_uint2(pack_bf16x2(wa * x.x + wb * y.x, wa * x.y + wb * y.y),
                                     pack_bf16x2(wa * x.z + wb * y.z, wa * x.w + wb * y.w));
        reinterpret_cast<uint2*>(o_out)[i] = out;
        if (c4 == 0) lse_out[row] = lse;
    }
}

// Pass B ("Cascade attention" page, second segment): virtual request
// v = b*topk + k attends only its own S draft tokens, draft s seeing drafts
// 0..s.  One warp per (v, query head): each lane holds 4 of the 128 head
// dimensions, scores are reduced across the warp with shuffles, and the
// softmax runs online (running max, rescaled sum and accumulator) over the
// visible drafts.
__global__ void __launch_bounds__(256) pass_b_kernel(PassBParams p) {
    const int warp_global = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int n_warps = p.B * p.topk * p.H_q;
    if (warp_global >= n_warps) return;
    const int v = warp_global / p.H_q;
    const int hq = warp_global % p.H_q;
    const int hk = hq / (p.H_q / p.H_kv);
    const int32_t* trow = p.dtab + (size_t)v * p.dtab_stride;
    for (int s = 0; s < p.S; ++s) {
        const size_t qoff = ((size_t)(v * p.S + s) * p.H_q + hq) * 128 + lane * 4;
        const uint2 qraw = __ldg(reinterpret_cast<const uint2*>(p.q + qoff));
        const float q0 = __uint_as_float(qraw.x << 16), q1 = __uint_as_float(qraw.x & 0xFFFF0000u);
        const float q2 = __uint_as_float(qraw.y << 16), q3 = __uint_as_float(qraw.y & 0xFFFF0000u);
        float m = ninf(), l = 0.f, a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
        for (int j = 0; j <= s; ++j) {
            const int pg = __ldg(trow + j / p.P);
            if (pg < 0 || pg >= p.num_pages) {
                if (lane == 0) atomicOr(p.status, CPA_DEV_BAD_PAGE);
                continue;
            }
            const size_t off = (((size_t)pg * p.P + (j % p.P)) * p.H_kv + hk) * 128 + lane * 4;
            const uint2 kr = __ldg(reinterpret_cast<const uint2*>(p.k_pages + off));
            const uint2 vr = __ldg(reinterpret_cast<const uint2*>(p.v_pages + off));
            float dot = q0 * __uint_as_float(kr.x << 16) + q1 * __uint_as_float(kr.x & 0xFFFF0000u) +
                        q2 * __uint_as_float(kr.y << 16) + q3 * __uint_as_float(kr.y & 0xFFFF0000u);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
            const float x = dot * p.scale_log2;
            const float m_new = fmaxf(m, x);
            const float c = ex2(m - m_new);  // 0 when m is -inf
            const float e = ex2(x - m_new);
            l = l * c + e;
            a0 = a0 * c + e * __uint_as_float(vr.x << 16);
            a1 = a1 * c + e * __uint_as_float(vr.x & 0xFFFF0000u);
            a2 = a2 * c + e * __uint_as_float(vr.y << 16);
            a3 = a3 * c + e * __uint_as_float(vr.y & 0xFFFF0000u);
            m = m_new;
        }
        const float inv = l > 0.f ? 1.f / l : 0.f;
        reinterpret_cast<float4*>(p.o_b + qoff)[0] = make_float4(a0 * inv, a1 * inv, a2 * inv, a3 * inv);
        if (lane == 0)
            p.lse_b[(size_t)(v * p.S + s) * p.H_q + hq] = l > 0.f ? (m + lg2(l)) * kLn2F : ninf();
    }
}

// Draft-tree pass (KV-cache tutorial, section 8.2 tip box on tree attention,
// and Q14): the N draft tokens of request b are a token tree flattened so that
// every parent precedes its children (BFS order does); node i sees tree node
// j iff j is i or one of i's ancestors.
//
// One CTA per (request, KV head).  It stages the request's N tree K/V rows of
// that head in shared memory (N <= 64 rows of 256 B each for K and for V),
// and builds each node's 64-bit ancestor-or-self mask by climbing the parent
// chain (at most N steps, as each step moves to a smaller index; a parent
// index outside [-1, i) stops the climb and sets CPA_DEV_BAD_TREE).  Then
// each warp takes (node, group of 4 query heads) tasks: a lane holds 4 of
// the 128 dimensions of the 4 heads' queries, and for every node in the mask
// (ascending) reads the K and V row from shared memory once for all 4 heads,
// reduces the 4 dot products across the warp with interleaved shuffles and
// updates 4 online softmaxes.  When the prefix pass's fp32 (o_a, lse_a) are
// given, the epilogue merges the two parts by the log-sum-exp identity of
// the cascade page and writes bf16 o; otherwise it writes its own fp32 part.
constexpr int kTreeHeadsPerWarp = 4;

__global__ void __launch_bounds__(256) tree_kernel(TreeParams p) {
    __shared__ __align__(16) __nv_bfloat16 ks[CPA_MAX_TREE_NODES][128];
    __shared__ __align__(16) __nv_bfloat16 vs[CPA_MAX_TREE_NODES][128];
    __shared__ unsigned long long anc_s[CPA_MAX_TREE_NODES];
    __shared__ unsigned long long rows_ok;  // bit j: row j came from a valid page
    const int b = blockIdx.x / p.H_kv, hk = blockIdx.x % p.H_kv;
    const int G = p.H_q / p.H_kv;
    const int32_t* trow = p.ttab + (size_t)b * p.ttab_stride;
    if (threadIdx.x == 0) rows_ok = 0ull;
    __syncthreads();
    // tree K/V rows of (b, hk), 16 bytes per thread and step
    for (int c = threadIdx.x; c < p.N * 16; c += blockDim.x) {
        const int j = c >> 4, part = c & 15;
        const int pg = __ldg(trow + j / p.P);
        uint4 kx = make_uint4(0u, 0u, 0u, 0u), vx = kx;
        if (pg >= 0 && pg < p.num_pages) {
            const size_t off = (((size_t)pg * p.P + (j % p.P)) * p.H_kv + hk) * 128 + part * 8;
            kx = __ldg(reinterpret_cast<const uint4*>(p.k_pages + off));
            vx = __ldg(reinterpret_cast<const uint4*>(p.v_pages + off));
            if (part == 0) atomicOr(&rows_ok, 1ull << j);
        } else if (part == 0) {
            atomicOr(p.status, CPA_DEV_BAD_PAGE);
        }
        reinterpret_cast<uint4*>(&ks[j][0])[part] = kx;
        reinterpret_cast<uint4*>(&vs[j][0])[part] = vx;
    }
    // ancestor-or-self masks
    const int32_t* par = p.parents + (size_t)b * p.N;
    for (int i = threadIdx.x; i < p.N; i += blockDim.x) {
        unsigned long long anc = 1ull << i;
        bool bad = false;
        for (int j = i, step = 0; step < p.N; ++step) {
            const int pj = __ldg(par + j);
            if (pj == -1) break;
            if (pj < -1 || pj >= j) {
                bad = true;
                break;
            }
            anc |= 1ull << pj;
            j = pj;
        }
        if (bad) atomicOr(p.status, CPA_DEV_BAD_TREE);
        anc_s[i] = anc;
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int groups = (G + kTreeHeadsPerWarp - 1) / kTreeHeadsPerWarp;
    const int n_tasks = p.N * groups;
    for (int task = threadIdx.x >> 5; task < n_tasks; task += blockDim.x >> 5) {
        const int i = task / groups;
        const int g0 = (task % groups) * kTreeHeadsPerWarp;
        const size_t tok = (size_t)b * p.N + i;
        float q[kTreeHeadsPerWarp][4], acc[kTreeHeadsPerWarp][4];
        float m[kTreeHeadsPerWarp], l[kTreeHeadsPerWarp];
#pragma unroll
        for (int u = 0; u < kTreeHeadsPerWarp; ++u) {
            uint2 qr = make_uint2(0u, 0u);
            if (g0 + u < G)
                qr = __ldg(reinterpret_cast<const uint2*>(
                    p.q + (tok * p.H_q + hk * G + g0 + u) * 128 + lane * 4));
            q[u][0] = __uint_as_float(qr.x << 16);
            q[u][1] = __uint_as_float(qr.x & 0xFFFF0000u);
            q[u][2] = __uint_as_float(qr.y << 16);
            q[u][3] = __uint_as_float(qr.y & 0xFFFF0000u);
            m[u] = ninf();
            l[u] = 0.f;
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[u][c] = 0.f;
        }
        for (unsigned long long rest = anc_s[i] & rows_ok; rest != 0ull; rest &= rest - 1ull) {
            const int j = __ffsll((long long)rest) - 1;
            const uint2 kr = reinterpret_cast<const uint2*>(&ks[j][0])[lane];
            const uint2 vr = reinterpret_cast<const uint2*>(&vs[j][0])[lane];
            const float k0 = __uint_as_float(kr.x << 16), k1 = __uint_as_float(kr.x & 0xFFFF0000u);
            const float k2 = __uint_as_float(kr.y << 16), k3 = __uint_as_float(kr.y & 0xFFFF0000u);
            const float v0 = __uint_as_float(vr.x << 16), v1 = __uint_as_float(vr.x & 0xFFFF0000u);
            const float v2 = __uint_as_float(vr.y << 16), v3 = __uint_as_float(vr.y & 0xFFFF0000u);
            float dot[kTreeHeadsPerWarp];
#pragma unroll
            for (int u = 0; u < kTreeHeadsPerWarp; ++u)
                dot[u] = q[u][0] * k0 + q[u][1] * k1 + q[u][2] * k2 + q[u][3] * k3;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
                for (int u = 0; u < kTreeHeadsPerWarp; ++u)
                    dot[u] += __shfl_xor_sync(0xffffffffu, dot[u], o);
            }
#pragma unroll
            for (int u = 0; u < kTreeHeadsPerWarp; ++u) {
                const float x = dot[u] * p.scale_log2;
                const float m_new = fmaxf(m[u], x);
                const float c = ex2(m[u] - m_new);  // 0 when m is -inf
                const float e = ex2(x - m_new);
                l[u] = l[u] * c + e;
                acc[u][0] = acc[u][0] * c + e * v0;
                acc[u][1] = acc[u][1] * c + e * v1;
                acc[u][2] = acc[u][2] * c + e * v2;
                acc[u][3] = acc[u][3] * c + e * v3;
                m[u] = m_new;
            }
        }
#pragma unroll
        for (int u = 0; u < kTreeHeadsPerWarp; ++u) {
            if (g0 + u >= G) continue;
            const size_t row = tok * p.H_q + hk * G + g0 + u;
            const size_t off = row * 128 + lane * 4;
            const float inv = l[u] > 0.f ? 1.f / l[u] : 0.f;
            const float lse_b = l[u] > 0.f ? (m[u] + lg2(l[u])) * kLn2F : ninf();
            const float b0 = acc[u][0] * inv, b1 = acc[u][1] * inv;
            const float b2 = acc[u][2] * inv, b3 = acc[u][3] * inv;
            if (p.o_a == nullptr) {
                reinterpret_cast<float4*>(static_cast<float*>(p.o) + off)[0] =
                    make_float4(b0, b1, b2, b3);
                if (lane == 0) p.lse[row] = lse_b;
                continue;
            }
            // merge with the prefix part about the larger log-sum-exp
            const float la = __ldg(p.lse_a + row);
            float wa, wb, lse;
            if (la == ninf() && lse_b == ninf()) {
                wa = 0.f;
                wb = 0.f;
                lse = ninf();
            } else {
                const float mx = fmaxf(la, lse_b);
                const float ea = ex2((la - mx) * kLog2eF), eb = ex2((lse_b - mx) * kLog2eF);
                const float s = ea + eb;
                wa = ea / s;
                wb = eb / s;
                lse = mx + lg2(s) * kLn2F;
            }
            const float4 x = __ldg(reinterpret_cast<const float4*>(p.o_a + off));
            reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.o) + off)[0] =
                make_uint2(pack_bf16x2(wa * x.x + wb * b0, wa * x.y + wb * b1),
                           pack_bf16x2(wa * x.z + wb * b2, wa * x.w + wb * b3));
            if (lane == 0) p.lse[row] = lse;
        }
    }
}

// Waits on a barrier that nothing completes; the bounded wait gives up after
// `limit_ns`, records CPA_DEV_TIMEOUT and the kernel returns normally.
__global__ void wait_timeout_kernel(uint32_t* status, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, status, limit_ns);
}

cudaError_t launch_merge_state(const float* o_a, const float* lse_a, const float* o_b,
                               const float* lse_b, long long n_rows, int head_dim, void* o_out,
                               float* lse_out, int n_sm, cudaStream_t stream) {
    const int d4 = head_dim / 4;
    const long long n = n_rows * d4;
    long long blocks = (n + 255) / 256;
    const long long cap = (long long)n_sm * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    merge_state_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
        o_a, lse_a, o_b, lse_b, n_rows, d4, static_cast<__nv_bfloat16*>(o_out), lse_out);
    return cudaGetLastError();
}

cudaError_t launch_pass_b(const PassBParams& p, cudaStream_t stream) {
    const long long warps = (long long)p.B * p.topk * p.H_q;
    const long long blocks = (warps + 7) / 8;
    pass_b_kernel<<<(unsigned)blocks, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_tree(const TreeParams& p, cudaStream_t stream) {
    const long long blocks = (long long)p.B * p.H_kv;
    tree_kernel<<<(unsigned)blocks, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_wait_timeout(uint32_t* status, unsigned long long limit_ns,
                                cudaStream_t stream) {
    wait_timeout_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
    return cudaGetLastError();
}

}  // namespace cpa
