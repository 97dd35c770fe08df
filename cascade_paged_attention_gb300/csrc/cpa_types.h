// cpa_types.h -- constants and the work-partition arithmetic shared by the
// host launcher and the kernels (compiled as both host and device code).
#pragma once
#include <stdint.h>

#include "cpa.h"

#if defined(__CUDACC__)
#define CPA_HD __host__ __device__ __forceinline__
#else
#define CPA_HD inline
#endif

namespace cpa {

// Keys per pipeline tile (one TMA stage, one N=128 QK^T MMA).
constexpr int kBN = 128;
// Draft tokens per branch of a verify unit (one draft tile holds every branch).
constexpr int kMaxDraft = 16;
// Rows of the partial-result slots (two 128-row M tiles).
constexpr int kMaxUnitRows = 256;

enum Mode : int {
    MODE_CASCADE = 0,       // Pass A (tensor cores) + fused Pass B + merge -> bf16 o
    MODE_NAIVE = 1,         // B*topk virtual requests, each over prefix + own drafts -> bf16 o
    MODE_PASS_A = 2,        // prefix only -> fp32 o_A, lse_A
    MODE_PREFILL = 3,       // prefix-hit prefill, rectangle + triangle -> bf16 o
    MODE_PREFILL_RECT = 4,  // rectangle only (keys 0..H-1) -> fp32
    MODE_PREFILL_TRI = 5,   // triangle only (keys H..H+i) -> fp32
    MODE_TREE = 6,          // Pass A + the draft tree as one masked tile + merge -> bf16 o
};

// Balanced contiguous split of `total` tiles over `n` CTAs:
// CTA c owns tiles [floor(c*T/n), floor((c+1)*T/n)).
// With fast32, a 32-bit division whenever total * n fits (a 64-bit division
// is a long software sequence on the GPU).  Both give the same result; the
// kernel instances choose the form that measured faster for them.
CPA_HD int64_t split_begin(int64_t total, int n, int c, bool fast32 = false) {
    if (fast32 && (uint64_t)total * (uint64_t)n < 0x80000000ull)
        return (int64_t)((uint32_t)total * (uint32_t)c / (uint32_t)n);
    return (total * c) / n;
}

// The CTA whose range holds tile x: the largest c with floor(c*T/n) <= x,
// which is ceil((x+1)*n/T) - 1.
CPA_HD int split_owner(int64_t total, int n, int64_t x, bool fast32 = false) {
    if (fast32 && (uint64_t)total * (uint64_t)n < 0x80000000ull)
        return (int)(((uint32_t)(x + 1) * (uint32_t)n - 1u) / (uint32_t)total);
    return (int)(((x + 1) * (int64_t)n - 1) / total);
}

// Partial-result slot of CTA c's piece of a unit that starts at tile
// u_start: slot 2c if that piece is the CTA's first piece of work, 2c+1 if
// the CTA began inside an earlier unit.  Only a CTA's first and last pieces
// can be split, so two slots per CTA suffice.
CPA_HD int split_slot(int64_t total, int n, int c, int64_t u_start, bool fast32 = false) {
    return 2 * c + ((split_begin(total, n, c, fast32) < u_start) ? 1 : 0);
}

}  // namespace cpa
