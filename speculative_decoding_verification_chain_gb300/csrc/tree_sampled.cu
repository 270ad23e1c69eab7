// tree_sampled.cu -- sampled token-tree verification on sm_103a.
//
// What it computes (EAGLE-3 review, "EAGLE-3 inference" step 4: with sampling,
// min(1, p/q) acceptance and residual correction keep the target
// distribution; the review's small-draft section gives A(x) = min(1, p/q) and
// the residual norm(max(0, p - q))).  The pages give no rule for siblings;
// the reading implemented: walk from the root; at node c, p' = softmax(z_c/T);
// test c's children in index order, child n (token x) accepted iff q_c(x) == 0
// or u_accept[n] < p'(x)/q_c(x); an accepted child becomes the next node; a
// rejected one replaces p' by norm(max(0, p' - q_c)) (kept if that has no
// mass); when no child is accepted, or c is a leaf, one token is drawn from p'
// by inverse CDF with u_sample[c].
//
// The j-fold residual is never formed step by step: since
// max(0, max(0, a) - b) = max(0, a - b) for b >= 0, after rejections with
// masses S_0 = 1, S_1, ..., p' is proportional to max(0, p - T q) with
// T = S_0 + ... + S_{j-1}, and S_j = sum max(0, p - T q).  Each rejection is
// then one pass over p and q of the row, both held in shared memory.
//
// Layout: one thread-block cluster per request; CTA r of the cluster holds
// columns [r * slice, (r + 1) * slice) of the current node's row (e = exp2 of
// the scaled logits, then q) in shared memory.  Scalars (row max, sums,
// masses, prefix sums) are combined across the cluster through distributed
// shared memory after a cluster barrier; every CTA runs the same control flow
// on the same combined values, so all of them take the same decisions.
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <climits>

#include "common.h"
#include "spec_verify.h"

namespace cg = cooperative_groups;

namespace sv {
namespace ts {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxNodes = SPEC_MAX_ROWS;       // N + 1
constexpr int kMaxCluster = 16;
constexpr int kSliceCap = 25600;               // columns per CTA: e and q (fp32) in 200 KiB
constexpr float kLog2e = 1.4426950408889634f;

struct Params {
    const void *logits;        // [B, N+1, V] bf16 bits or fp32
    const float *q;            // [B, N+1, V]
    const int32_t *tokens;     // [B, N]
    const float *temperature;  // [B]
    const float *u_accept;     // [B, N]
    const float *u_sample;     // [B, N+1]
    int32_t *out_path;         // [B, D+1]
    int32_t *out_tokens;       // [B, D+1]
    int32_t *out_len;          // [B]
    int32_t *status;           // one word or null
    int bf16, B, N, V, max_depth, slice, cluster, vec_z, vec_q;
    uint16_t child_off[kMaxNodes + 1];  // children of c: child_list[child_off[c] .. child_off[c+1])
    uint8_t child_list[kMaxNodes];
};

struct Shared {
    double slot[2][2];          // cluster exchange, double-buffered by reduction parity
    double wsum[kWarps];
    float wmax[kWarps];
    int wint[2][kWarps];
    int dec;
};

// ---------------------------------------------------------------- helpers --
__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }

// Compensated (Neumaier) running sum in fp32: s + c is the sum to ~1 ulp of
// the terms' magnitude, whatever the chunk length.
__device__ __forceinline__ void nadd(float &s, float &c, float v) {
    const float t = s + v;
    const bool big = fabsf(s) >= fabsf(v);
    c += big ? (s - t) + v : (v - t) + s;
    s = t;
}

__device__ __forceinline__ double block_sum(double v, Shared &sh) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) sh.wsum[w] = v;
    __syncthreads();
    double r = 0.0;
    for (int i = 0; i < kWarps; ++i) r += sh.wsum[i];
    __syncthreads();
    return r;
}

__device__ __forceinline__ float block_max(float v, Shared &sh) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) sh.wmax[w] = v;
    __syncthreads();
    float r = -INFINITY;
    for (int i = 0; i < kWarps; ++i) r = fmaxf(r, sh.wmax[i]);
    __syncthreads();
    return r;
}

// Block minimum of a and maximum of b (ints).
__device__ __forceinline__ void block_minmax(int &a, int &b, Shared &sh) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        a = min(a, __shfl_xor_sync(0xffffffffu, a, o));
        b = max(b, __shfl_xor_sync(0xffffffffu, b, o));
    }
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        sh.wint[0][w] = a;
        sh.wint[1][w] = b;
    }
    __syncthreads();
    a = INT_MAX;
    b = -1;
    for (int i = 0; i < kWarps; ++i) {
        a = min(a, sh.wint[0][i]);
        b = max(b, sh.wint[1][i]);
    }
    __syncthreads();
}

// Exclusive prefix over the block's threads (thread order) of v; *total gets
// the block sum.
__device__ __forceinline__ double block_excl_scan(double v, double *total, Shared &sh) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    double x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh.wsum[w] = x;
    __syncthreads();
    double before = 0.0, all = 0.0;
    for (int i = 0; i < kWarps; ++i) {
        if (i < w) before += sh.wsum[i];
        all += sh.wsum[i];
    }
    __syncthreads();
    *total = all;
    return before + x - v;
}

// Calls f(r, a_r, b_r) for every rank r in rank order after one cluster
// barrier; (a, b) are this CTA's values (thread 0's).  The two parity slots
// make a second barrier unnecessary: a slot is rewritten only after every CTA
// has passed the barrier that follows its last read of it.
template <class F>
__device__ __forceinline__ void cluster_each(cg::cluster_group &cl, Shared &sh, int &parity, double a, double b,
                                             int C, F f) {
    if (threadIdx.x == 0) {
        sh.slot[parity][0] = a;
        sh.slot[parity][1] = b;
    }
    cl.sync();
    for (int r = 0; r < C; ++r) {
        const double *rem = cl.map_shared_rank(&sh.slot[parity][0], r);
        f(r, rem[0], rem[1]);
    }
    parity ^= 1;
}

__device__ __forceinline__ bool nonfinite(float f) { return (f != f) || f == INFINITY; }

// Columns [lo, lo + n) of one logits row (element offset roff) into dst as
// fp32; returns this thread's maximum and ORs NaN / +inf into bad.
__device__ float load_logits(const Params &P, size_t roff, int lo, int n, float *dst, bool &bad) {
    float m = -INFINITY;
    if (P.bf16) {
        const uint16_t *src = static_cast<const uint16_t *>(P.logits) + roff + lo;
        int done = 0;
        if (P.vec_z) {
            const int nv = n >> 3;
            const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
            for (int i = threadIdx.x; i < nv; i += kThreads) {
                const uint4 v = __ldg(s4 + i);
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                float f[8];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    f[2 * j] = __uint_as_float(w[j] << 16);
                    f[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    m = fmaxf(m, f[j]);
                    bad |= nonfinite(f[j]);
                }
                float4 *d4 = reinterpret_cast<float4 *>(dst + 8 * i);
                d4[0] = make_float4(f[0], f[1], f[2], f[3]);
                d4[1] = make_float4(f[4], f[5], f[6], f[7]);
            }
            done = nv << 3;
        }
        for (int i = done + threadIdx.x; i < n; i += kThreads) {
            const float f = bf16_to_f32(__ldg(src + i));
            m = fmaxf(m, f);
            bad |= nonfinite(f);
            dst[i] = f;
        }
    } else {
        const float *src = static_cast<const float *>(P.logits) + roff + lo;
        int done = 0;
        if (P.vec_z) {
            const int nv = n >> 2;
            const float4 *s4 = reinterpret_cast<const float4 *>(src);
            for (int i = threadIdx.x; i < nv; i += kThreads) {
                const float4 v = __ldg(s4 + i);
                m = fmaxf(fmaxf(m, fmaxf(v.x, v.y)), fmaxf(v.z, v.w));
                bad |= nonfinite(v.x) | nonfinite(v.y) | nonfinite(v.z) | nonfinite(v.w);
                reinterpret_cast<float4 *>(dst)[i] = v;
            }
            done = nv << 2;
        }
        for (int i = done + threadIdx.x; i < n; i += kThreads) {
            const float f = __ldg(src + i);
            m = fmaxf(m, f);
            bad |= nonfinite(f);
            dst[i] = f;
        }
    }
    return m;
}

// Columns [lo, lo + n) of one q row (element offset roff) into dst.
__device__ void load_q(const Params &P, size_t roff, int lo, int n, float *dst) {
    const float *src = P.q + roff + lo;
    int done = 0;
    if (P.vec_q) {
        const int nv = n >> 2;
        const float4 *s4 = reinterpret_cast<const float4 *>(src);
        for (int i = threadIdx.x; i < nv; i += kThreads) reinterpret_cast<float4 *>(dst)[i] = __ldg(s4 + i);
        done = nv << 2;
    }
    for (int i = done + threadIdx.x; i < n; i += kThreads) dst[i] = __ldg(src + i);
}

__global__ void __launch_bounds__(kThreads, 1) tree_sampled_kernel(const __grid_constant__ Params P) {
    extern __shared__ __align__(16) float dyn[];
    __shared__ Shared sh;
    cg::cluster_group cl = cg::this_cluster();
    const int C = P.cluster;
    const int rank = static_cast<int>(cl.block_rank());
    const int b = static_cast<int>(blockIdx.x) / C;
    const int S = P.slice, V = P.V, N = P.N, D1 = P.max_depth + 1;
    float *ev = dyn;        // e = exp2((z - M) * log2(e) / T) of this CTA's columns
    float *qv = dyn + S;    // q of this CTA's columns (loaded on the first rejection at a node)
    const int lo = rank * S;
    const int n = max(0, min(S, V - lo));
    // Thread t owns the contiguous chunk [t*E, t*E + E) of the CTA's columns;
    // E is odd so that consecutive threads fall in different banks.
    const int E = ((n + kThreads - 1) / kThreads) | 1;
    const int c0 = min(n, static_cast<int>(threadIdx.x) * E), c1 = min(n, c0 + E);
    const bool lead = rank == 0 && threadIdx.x == 0;
    int parity = 0;
    bool bad = false;

    float T = __ldg(P.temperature + b);
    if (!(T > 0.0f) || T == INFINITY) {
        if (lead && P.status) atomicOr(P.status, SPEC_STATUS_BAD_TEMPERATURE);
        T = 1.0f;
    }
    const float c2 = kLog2e / T;
    const size_t rows = static_cast<size_t>(N) + 1;
    if (lead) P.out_path[static_cast<size_t>(b) * D1] = 0;

    int cur = 0, d = 0;
    for (;;) {
        const size_t roff = (static_cast<size_t>(b) * rows + cur) * static_cast<size_t>(V);
        // row max over the cluster
        float m = block_max(load_logits(P, roff, lo, n, ev, bad), sh);
        float M = -INFINITY;
        cluster_each(cl, sh, parity, static_cast<double>(m), 0.0, C,
                     [&](int, double a, double) { M = fmaxf(M, static_cast<float>(a)); });
        // e and its sum (rank order, so every CTA holds the same value)
        float s = 0.0f, c = 0.0f;
        for (int i = c0; i < c1; ++i) {
            const float e = exp2f((ev[i] - M) * c2);
            ev[i] = e;
            nadd(s, c, e);
        }
        const double part = block_sum(static_cast<double>(s) + static_cast<double>(c), sh);
        double Ssum = 0.0;
        cluster_each(cl, sh, parity, part, 0.0, C, [&](int, double a, double) { Ssum += a; });
        if (!(Ssum > 0.0) || !(Ssum < INFINITY)) {
            bad = true;
            Ssum = 1.0;
        }
        const double invS = 1.0 / Ssum;
        const float invSf = static_cast<float>(invS);

        // children in index order; (Tm, ST): p' is max(0, p - Tm q) / ST
        double Tm = 0.0, ST = 1.0;
        bool qloaded = false;
        int next = -1;
        for (int k = P.child_off[cur]; k < P.child_off[cur + 1]; ++k) {
            const int nd = P.child_list[k];
            if (threadIdx.x == 0) {
                const int x = __ldg(P.tokens + static_cast<size_t>(b) * N + (nd - 1));
                int acc = 0;
                if (x < 0 || x >= V) {
                    if (rank == 0 && P.status) atomicOr(P.status, SPEC_STATUS_TOKEN_RANGE);
                } else {
                    const int owner = x / S;
                    const float ex = *cl.map_shared_rank(ev + (x - owner * S), owner);
                    const double qx = static_cast<double>(__ldg(P.q + roff + x));
                    if (qx == 0.0) {
                        acc = 1;
                    } else {
                        double r = static_cast<double>(ex) * invS - Tm * qx;
                        r = r > 0.0 ? r : 0.0;
                        const double u = static_cast<double>(__ldg(P.u_accept + static_cast<size_t>(b) * N + (nd - 1)));
                        acc = u < r / (ST * qx);
                    }
                }
                sh.dec = acc;
            }
            __syncthreads();
            const int acc = sh.dec;
            __syncthreads();
            if (acc) {
                next = nd;
                break;
            }
            // rejected: p' <- norm(max(0, p' - q)), i.e. Tm <- Tm + ST and ST <- its mass
            if (!qloaded) {
                load_q(P, roff, lo, n, qv);
                __syncthreads();
                qloaded = true;
            }
            const double Tn = Tm + ST;
            const float Tnf = static_cast<float>(Tn);
            s = 0.0f;
            c = 0.0f;
            for (int i = c0; i < c1; ++i) nadd(s, c, fmaxf(0.0f, fmaf(-Tnf, qv[i], ev[i] * invSf)));
            const double rpart = block_sum(static_cast<double>(s) + static_cast<double>(c), sh);
            double Sn = 0.0;
            cluster_each(cl, sh, parity, rpart, 0.0, C, [&](int, double a, double) { Sn += a; });
            if (Sn > 0.0) {  // a residual of no mass leaves p' as it is
                Tm = Tn;
                ST = Sn;
            }
        }
        if (next < 0) {
            // one draw from p' (weights e, or max(0, e/S - Tm q) after a
            // rejection): the smallest column whose prefix sum exceeds
            // t = u * (total); the prefix runs over CTAs in rank order, threads
            // in thread order and columns in index order, all in the same
            // compensated sums, so the total and the prefixes agree.
            const bool resid = Tm > 0.0;
            const float Tf = static_cast<float>(Tm);
            s = 0.0f;
            c = 0.0f;
            int lastpos = -1;
            for (int i = c0; i < c1; ++i) {
                const float w = resid ? fmaxf(0.0f, fmaf(-Tf, qv[i], ev[i] * invSf)) : ev[i];
                nadd(s, c, w);
                if (w > 0.0f) lastpos = lo + i;
            }
            double btot = 0.0;
            const double texcl = block_excl_scan(static_cast<double>(s) + static_cast<double>(c), &btot, sh);
            double cexcl = 0.0, total = 0.0;
            cluster_each(cl, sh, parity, btot, 0.0, C, [&](int r, double a, double) {
                if (r < rank) cexcl += a;
                total += a;
            });
            const double t = static_cast<double>(__ldg(P.u_sample + static_cast<size_t>(b) * rows + cur)) * total;
            const double base = cexcl + texcl;
            int cand = INT_MAX;
            if (c1 > c0 && base <= t) {
                float s2 = 0.0f, k2 = 0.0f;
                for (int i = c0; i < c1; ++i) {
                    const float w = resid ? fmaxf(0.0f, fmaf(-Tf, qv[i], ev[i] * invSf)) : ev[i];
                    nadd(s2, k2, w);
                    if (base + (static_cast<double>(s2) + static_cast<double>(k2)) > t) {
                        cand = lo + i;
                        break;
                    }
                }
            }
            block_minmax(cand, lastpos, sh);
            int pick = INT_MAX, last = -1;
            cluster_each(cl, sh, parity, static_cast<double>(cand), static_cast<double>(lastpos), C,
                         [&](int, double a, double l) {
                             pick = min(pick, static_cast<int>(a));
                             last = max(last, static_cast<int>(l));
                         });
            if (pick == INT_MAX) pick = last >= 0 ? last : V - 1;  // t at or past the total after rounding
            if (lead) {
                int32_t *ot = P.out_tokens + static_cast<size_t>(b) * D1;
                int32_t *op = P.out_path + static_cast<size_t>(b) * D1;
                ot[d] = pick;
                for (int i = d + 1; i < D1; ++i) {
                    ot[i] = -1;
                    op[i] = -1;
                }
                P.out_len[b] = d + 1;
            }
            break;
        }
        if (lead) {
            P.out_tokens[static_cast<size_t>(b) * D1 + d] = __ldg(P.tokens + static_cast<size_t>(b) * N + (next - 1));
            P.out_path[static_cast<size_t>(b) * D1 + d + 1] = next;
        }
        ++d;
        cur = next;
        cl.sync();  // every remote read of this row's e is done before any CTA loads the next row
    }
    if (bad && P.status) atomicOr(P.status, SPEC_STATUS_NONFINITE);
    cl.sync();  // keep this CTA's shared memory alive until the last remote read of it
}

}  // namespace ts

namespace {

struct TsDevice {
    int ok = 0;
};
TsDevice g_ts_dev[64];

spec_status_t ts_setup() {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    int sms = 0;
    spec_status_t st = require_sm103(&sms);
    if (st != SPEC_OK) return st;
    if (dev < 0 || dev >= 64) return fail(SPEC_ERR_UNSUPPORTED, "device index out of range%s");
    if (!g_ts_dev[dev].ok) {
        const void *k = reinterpret_cast<const void *>(ts::tree_sampled_kernel);
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(2 * sizeof(float) * ts::kSliceCap));
        if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "sampled tree kernel setup: %s", cudaGetErrorString(e));
        g_ts_dev[dev].ok = 1;
    }
    return SPEC_OK;
}

inline int round8(long long x) { return static_cast<int>((x + 7) / 8 * 8); }

}  // namespace
}  // namespace sv

extern "C" spec_status_t spec_verify_tree_sampled(const void *target_logits, spec_dtype_t dtype,
                                                  const float *draft_probs, const int32_t *node_tokens,
                                                  const int32_t *parent, const float *temperature,
                                                  const float *u_accept, const float *u_sample, int B, int N, int V,
                                                  int max_depth, int32_t *out_path, int32_t *out_tokens,
                                                  int32_t *out_len, int32_t *d_status, void *stream) {
    using namespace sv;
    if (B < 1 || N < 0 || N > SPEC_MAX_ROWS - 1 || V < 1 || max_depth < 0 || max_depth > SPEC_MAX_ROWS - 1)
        return fail(SPEC_ERR_INVALID_ARG, "need B >= 1, 0 <= N <= 255, V >= 1, 0 <= max_depth <= 255%s");
    if (dtype != SPEC_BF16 && dtype != SPEC_FP32) return fail(SPEC_ERR_INVALID_ARG, "unknown dtype%s");
    if (!target_logits || !parent || !temperature || !u_sample || !out_path || !out_tokens || !out_len)
        return fail(SPEC_ERR_INVALID_ARG, "a required pointer is NULL%s");
    if (N > 0 && (!draft_probs || !node_tokens || !u_accept))
        return fail(SPEC_ERR_INVALID_ARG, "draft_probs, node_tokens and u_accept are required when N > 0%s");
    if (reinterpret_cast<uintptr_t>(target_logits) % 16 != 0 || reinterpret_cast<uintptr_t>(draft_probs) % 16 != 0)
        return fail(SPEC_ERR_INVALID_ARG, "target_logits and draft_probs must be 16-byte aligned%s");
    ts::Params P;
    memset(&P, 0, sizeof P);
    if (parent[0] != -1) return fail(SPEC_ERR_INVALID_ARG, "parent[0] must be -1%s");
    int depth[ts::kMaxNodes];
    int cnt[ts::kMaxNodes + 1];
    depth[0] = 0;
    for (int c = 0; c <= N + 1; ++c) cnt[c] = 0;
    for (int n = 1; n <= N; ++n) {
        if (parent[n] < 0 || parent[n] >= n) return fail(SPEC_ERR_INVALID_ARG, "need 0 <= parent[n] < n%s");
        depth[n] = depth[parent[n]] + 1;
        if (depth[n] > max_depth) return fail(SPEC_ERR_INVALID_ARG, "max_depth is below the tree's depth%s");
        cnt[parent[n] + 1]++;
    }
    for (int c = 0; c <= N; ++c) cnt[c + 1] += cnt[c];
    for (int c = 0; c <= N + 1; ++c) P.child_off[c] = static_cast<uint16_t>(cnt[c]);
    for (int n = 1; n <= N; ++n) P.child_list[cnt[parent[n]]++] = static_cast<uint8_t>(n);  // index order per parent
    int C = 1;
    while (C < ts::kMaxCluster && round8((V + C - 1) / C) > ts::kSliceCap) C *= 2;
    while (C < 8 && round8((V + C - 1) / C) > 4096) C *= 2;
    const int S = round8((V + C - 1) / C);
    if (S > ts::kSliceCap) return fail(SPEC_ERR_INVALID_ARG, "V is above 409600 (16 CTAs x 25600 columns)%s");
    spec_status_t st = ts_setup();
    if (st != SPEC_OK) return st;
    const int es = dtype == SPEC_BF16 ? 2 : 4;
    P.logits = target_logits;
    P.q = draft_probs;
    P.tokens = node_tokens;
    P.temperature = temperature;
    P.u_accept = u_accept;
    P.u_sample = u_sample;
    P.out_path = out_path;
    P.out_tokens = out_tokens;
    P.out_len = out_len;
    P.status = d_status;
    P.bf16 = dtype == SPEC_BF16;
    P.B = B;
    P.N = N;
    P.V = V;
    P.max_depth = max_depth;
    P.slice = S;
    P.cluster = C;
    P.vec_z = (static_cast<long long>(V) * es) % 16 == 0;
    P.vec_q = V % 4 == 0;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(static_cast<unsigned>(B) * static_cast<unsigned>(C));
    cfg.blockDim = dim3(ts::kThreads);
    cfg.dynamicSmemBytes = 2 * sizeof(float) * static_cast<size_t>(S);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(C);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, ts::tree_sampled_kernel, P);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "sampled tree launch: %s", cudaGetErrorString(e));
    return SPEC_OK;
}
