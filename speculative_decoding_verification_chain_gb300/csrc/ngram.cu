// ngram.cu -- n-gram lookup drafting on sm_103a.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.h"
#include "spec_verify.h"

namespace sv {

// ---------------------------------------------------------- n-gram lookup --
// Draft proposal without a model (serving-book chapter, draft sources, "n-gram
// lookup"): the longest n in [n_min, n_max] whose ending s[L-n..L-1] occurs
// ending earlier, at e < L-1; the latest such e; the draft is s[e+1..], at
// most k tokens.  One block per sequence: each thread takes ends e and counts
// how far s[e], s[e-1], ... agree with the ending (kept in shared memory);
// the block keeps the largest (match length, e).
constexpr int kNgramMax = 64;
constexpr int kNgramThreads = 1024;
constexpr int kNgramBatch = 8;

__global__ void __launch_bounds__(kNgramThreads) ngram_kernel(const int32_t *tokens, const int32_t *lengths, int Lmax,
                                                              int n_min, int n_max, int k, int32_t *out_draft,
                                                              int32_t *out_count, int32_t *out_len, int32_t *out_end) {
    __shared__ int32_t tail[kNgramMax];
    __shared__ unsigned long long wbest[kNgramThreads / 32];
    const int b = blockIdx.x;
    const int32_t *s = tokens + static_cast<size_t>(b) * Lmax;
    const int L = min(max(__ldg(lengths + b), 0), Lmax);
    for (int t = threadIdx.x; t < n_max; t += blockDim.x) tail[t] = (L - 1 - t >= 0) ? __ldg(s + L - 1 - t) : 0;
    __syncthreads();
    unsigned long long best = 0;   // (match length << 32) | (e + 1); 0: none
    const int32_t last = L > 0 ? tail[0] : 0;
    // kNgramBatch independent loads of s[e] per thread before any branch on
    // them; only ends whose token equals the last one extend the comparison.
    for (int e0 = L - 2 - static_cast<int>(threadIdx.x); e0 >= n_min - 1; e0 -= kNgramBatch * kNgramThreads) {
        int32_t v[kNgramBatch];
#pragma unroll
        for (int u = 0; u < kNgramBatch; ++u) {
            const int e = e0 - u * kNgramThreads;
            v[u] = e >= n_min - 1 ? __ldg(s + e) : ~last;
        }
#pragma unroll
        for (int u = 0; u < kNgramBatch; ++u) {
            if (v[u] != last) continue;
            const int e = e0 - u * kNgramThreads;
            int m = 1;
            while (m < n_max && m <= e && __ldg(s + e - m) == tail[m]) ++m;
            if (m >= n_min) {
                const unsigned long long key = (static_cast<unsigned long long>(m) << 32) | static_cast<unsigned>(e + 1);
                best = key > best ? key : best;
            }
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, off);
        best = o > best ? o : best;
    }
    if ((threadIdx.x & 31) == 0) wbest[threadIdx.x >> 5] = best;
    __syncthreads();
    if (threadIdx.x < 32) {
        best = threadIdx.x < kNgramThreads / 32 ? wbest[threadIdx.x] : 0;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, off);
            best = o > best ? o : best;
        }
        if (threadIdx.x == 0) wbest[0] = best;
    }
    __syncthreads();
    best = wbest[0];
    const int m = static_cast<int>(best >> 32);
    const int e = static_cast<int>(best & 0xffffffffull) - 1;
    for (int j = threadIdx.x; j < k; j += blockDim.x)
        out_draft[static_cast<size_t>(b) * k + j] = (e >= 0 && e + 1 + j < L) ? __ldg(s + e + 1 + j) : -1;
    if (threadIdx.x == 0) {
        out_count[b] = e >= 0 ? min(k, L - 1 - e) : 0;
        if (out_len) out_len[b] = m;
        if (out_end) out_end[b] = e;
    }
}

}  // namespace sv

using namespace sv;

extern "C" spec_status_t spec_ngram_propose(const int32_t *tokens, const int32_t *lengths, int B, int Lmax,
                                            int n_min, int n_max, int k, int32_t *out_draft, int32_t *out_count,
                                            int32_t *out_match_len, int32_t *out_match_end, void *stream) {
    clear_error();
    if (B < 0 || Lmax < 0 || n_min < 1 || n_max < n_min || n_max > kNgramMax || k < 0)
        return fail(SPEC_ERR_INVALID_ARG, "sizes out of range (B, Lmax >= 0; 1 <= n_min <= n_max <= 64; k >= 0)%s");
    if (B == 0) return SPEC_OK;
    if ((Lmax > 0 && !tokens) || !lengths || (k > 0 && !out_draft) || !out_count)
        return fail(SPEC_ERR_INVALID_ARG, "a required pointer is NULL%s");
    ngram_kernel<<<static_cast<unsigned>(B), kNgramThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        tokens, lengths, Lmax, n_min, n_max, k, out_draft, out_count, out_match_len, out_match_end);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "n-gram launch: %s", cudaGetErrorString(e));
    return SPEC_OK;
}
