// cpa_small.h -- launchers of the light kernels (merge_state, Pass B, the
// bounded-wait check), implemented in cpa_small.cu.
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

cudaError_t launch_merge_state(const float* o_a, const float* lse_a, const float* o_b,
                               const float* lse_b, long long n_rows, int head_dim, void* o_out,
                               float* lse_out, int n_sm, cudaStream_t stream);
cudaError_t launch_pass_b(const PassBParams& p, cudaStream_t stream);
cudaError_t launch_wait_timeout(uint32_t* status, unsigned long long limit_ns,
                                cudaStream_t stream);

}  // namespace cpa
