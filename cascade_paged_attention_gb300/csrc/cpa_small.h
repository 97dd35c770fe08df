// cpa_small.h -- launchers of the light kernels (merge_state, Pass B, the
// draft-tree pass, the bounded-wait check), implemented in cpa_small.cu.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace cpa {

struct PassBParams {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k_pages;
    const __nv_bfloat16* v_pages;
    const int32_t* dtab;
    int dtab_stride;
    int B, topk, S, H_q, H_kv, P, num_pages;
    float scale_log2;
    float* o_b;
    float* lse_b;
    uint32_t* status;
};

// Draft-tree pass: node i of request b (token b*N + i) against the tree
// nodes of its ancestor-or-self set.  With o_a / lse_a set it also merges the
// prefix pass's fp32 partial into a bf16 output; without, it writes its own
// fp32 partial.
struct TreeParams {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k_pages;
    const __nv_bfloat16* v_pages;
    const int32_t* ttab;     // [B, ttab_stride] page ids of the tree tokens
    int ttab_stride;
    const int32_t* parents;  // [B, N], -1 for a root, parents[i] < i otherwise
    int B, N, H_q, H_kv, P, num_pages;
    float scale_log2;
    const float* o_a;        // fp32 [B*N, H_q, 128] or null
    const float* lse_a;      // fp32 [B*N, H_q] (natural log) or null
    void* o;                 // bf16 when merging, fp32 otherwise
    float* lse;
    uint32_t* status;
};

cudaError_t launch_merge_state(const float* o_a, const float* lse_a, const float* o_b,
                               const float* lse_b, long long n_rows, int head_dim, void* o_out,
                               float* lse_out, int n_sm, cudaStream_t stream);
cudaError_t launch_pass_b(const PassBParams& p, cudaStream_t stream);
cudaError_t launch_tree(const TreeParams& p, cudaStream_t stream);
cudaError_t launch_wait_timeout(uint32_t* status, unsigned long long limit_ns,
                                cudaStream_t stream);

}  // namespace cpa
