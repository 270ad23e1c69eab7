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
// columns [r * slice, (r + 1) * slice) of the current node's row in shared
// memory: the logits as stored (one bulk-async copy), e = 2^((z - M) log2e/T)
// in fp32, and q (a second bulk copy, issued with the first whenever the node
// has children).  Values are combined across the cluster by exchanges: each
// CTA pushes one float4 (its max with its sum, a residual mass, a chunk
// total) into a slot of every CTA with st.async, completing on that CTA's
// own mbarrier, and each CTA reads the C slots in rank order, so every CTA
// holds the same numbers and takes the same decisions.  The row max and sum
// share one exchange: a CTA's sum is taken against its own max m_r and
// rescaled by 2^((m_r - M) log2e/T) afterwards.  The CTA owning a child's
// column pushes that child's e(x) with the same exchange.
// All arithmetic is fp32: a thread's few running sums are plain fp32 and
// every combination beyond a thread is two-float (about 44 significant
// bits); FP64 issue is scarce on this part and its latency sits on the
// walk's critical path.
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <climits>

#include "common.h"
#include "ptx.cuh"
#include "spec_verify.h"
#include "twofloat.cuh"

namespace cg = cooperative_groups;

namespace sv {
namespace ts {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxNodes = SPEC_MAX_ROWS;            // N + 1
constexpr int kMaxCluster = 16;
constexpr int kSmemBudget = 220 * 1024;             // dynamic: e, q (fp32) and the logits slice as stored
constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned long long kWaitLimitNs = 500000000ull;   // 0.5 s: the limit on copies in flight at exit

// Columns per CTA for a logits element of es bytes (8 + es bytes a column).
__host__ __device__ constexpr int slice_cap(int es) { return (kSmemBudget / (8 + es)) & ~7; }

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
    int bf16, B, N, V, max_depth, slice, cluster;
    int zbulk, qbulk;          // rows start on 16-byte boundaries: bulk copies allowed
    unsigned long long wait_ns;  // limit of the row-copy and cluster-exchange waits
    uint16_t child_off[kMaxNodes + 1];  // children of c: child_list[child_off[c] .. child_off[c+1])
    uint8_t child_list[kMaxNodes];
};

struct Shared {
    uint64_t bar;                          // the current node's row copies
    uint64_t xbar[2];                      // cluster exchanges, by exchange parity
    float4 slot[2][kMaxCluster];           // pushed by every rank, double-buffered by exchange parity
    float ws[kWarps], wc[kWarps];          // warp partials (two-float)
    float wxs[kWarps], wxc[kWarps];        // warp exclusive prefixes (two-float, final draw)
    float tot[2];                          // block total (final draw)
    float wmax[kWarps];
    int wint[kWarps];
    int dec;
    int pick;
    int32_t tok[kMaxNodes];                // node tokens of this request (node n at n-1)
    float ua[kMaxNodes];                   // u_accept of this request (node n at n-1)
    float qx[kMaxNodes];                   // q_c(x) of the current node's children, in child order
    float fr[kMaxCluster];                 // per-rank scale 2^((m_r - M) c2) of the current row (thread 0)
    float exb[2][kMaxNodes];               // e(x) of the same on the owner's own scale, pushed by the
                                           // owner; double-buffered by the parity of the node's depth
};

// ---------------------------------------------------------------- helpers --
__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }

// 2^x by the SFU approximation (relative error about 2^-22).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Kahan running sum of non-negative terms: s - c carries the sum to about one
// ulp of its magnitude, whatever the chunk length.
__device__ __forceinline__ void kadd(float &s, float &c, float v) {
    const float y = v - c;
    const float t = s + y;
    c = (t - s) - y;
    s = t;
}

// Two-float helpers on split (hi, lo) registers, over the shared two-float
// arithmetic.
__device__ __forceinline__ void tf_add(float &hi, float &lo, float bh, float bl) {
    const tf r = sv::tf_add(tf{hi, lo}, tf{bh, bl});
    hi = r.h;
    lo = r.l;
}

__device__ __forceinline__ void tf_mul(float ah, float al, float f, float &hi, float &lo) {
    const tf r = tf_mulf(tf{ah, al}, f);
    hi = r.h;
    lo = r.l;
}

// Block sum of the threads' two-float values; warp 0 combines the warps; the
// result reaches every thread.
__device__ __forceinline__ void block_sum2(float &hi, float &lo, Shared &sh) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        tf_add(hi, lo, __shfl_xor_sync(0xffffffffu, hi, o), __shfl_xor_sync(0xffffffffu, lo, o));
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        sh.ws[w] = hi;
        sh.wc[w] = lo;
    }
    __syncthreads();
    if (w == 0) {
        hi = lane < kWarps ? sh.ws[lane] : 0.0f;
        lo = lane < kWarps ? sh.wc[lane] : 0.0f;
#pragma unroll
        for (int o = kWarps / 2; o > 0; o >>= 1)
            tf_add(hi, lo, __shfl_xor_sync(0xffffffffu, hi, o), __shfl_xor_sync(0xffffffffu, lo, o));
        if (lane == 0) {
            sh.tot[0] = hi;
            sh.tot[1] = lo;
        }
    }
    __syncthreads();
    hi = sh.tot[0];
    lo = sh.tot[1];
}

__device__ __forceinline__ float block_max(float v, Shared &sh) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) sh.wmax[w] = v;
    __syncthreads();
    v = sh.wmax[lane & (kWarps - 1)];
#pragma unroll
    for (int o = kWarps / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Block maximum of an int, to every thread.
__device__ __forceinline__ int block_imax(int v, Shared &sh) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) sh.wint[w] = v;
    __syncthreads();
    v = sh.wint[lane & (kWarps - 1)];
#pragma unroll
    for (int o = kWarps / 2; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Exclusive and inclusive prefixes, in thread order, of the threads'
// two-float values.  Consecutive threads' boundaries are the same numbers (the
// same operations in the same order), and so is the last inclusive prefix and
// the block total, which goes to (th, tl).
__device__ __forceinline__ void block_scan2(float s, float c, float &exh, float &exl, float &inh, float &inl,
                                            float &th, float &tl, Shared &sh) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    float is = s, ic = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float ys = __shfl_up_sync(0xffffffffu, is, o), yc = __shfl_up_sync(0xffffffffu, ic, o);
        if (lane >= o) {
            float h = ys, l = yc;
            tf_add(h, l, is, ic);
            is = h;
            ic = l;
        }
    }
    float es = __shfl_up_sync(0xffffffffu, is, 1), ec = __shfl_up_sync(0xffffffffu, ic, 1);
    if (lane == 0) es = ec = 0.0f;
    if (lane == 31) {
        sh.ws[w] = is;
        sh.wc[w] = ic;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float h = 0.0f, l = 0.0f;
        for (int i = 0; i < kWarps; ++i) {
            sh.wxs[i] = h;
            sh.wxc[i] = l;
            tf_add(h, l, sh.ws[i], sh.wc[i]);
        }
        sh.tot[0] = h;
        sh.tot[1] = l;
    }
    __syncthreads();
    exh = sh.wxs[w];
    exl = sh.wxc[w];
    inh = exh;
    inl = exl;
    if (lane > 0) tf_add(exh, exl, es, ec);
    tf_add(inh, inl, is, ic);
    th = sh.tot[0];
    tl = sh.tot[1];
}

// Exchange number xk: every CTA sends its float4 into slot[xk & 1][its rank]
// of every CTA (threads 0..C-1, one st.async each) and waits on its own
// barrier xbar[xk & 1] (phase (xk >> 1) & 1) for C such stores plus `extra`
// bytes of other pushes tied to this exchange; then every thread reads the C
// local slots.  A slot or barrier phase is reused two exchanges later: a CTA
// sends exchange xk + 2 only after receiving every CTA's exchange xk + 1, and
// every CTA passes a block barrier between reading exchange xk and sending
// xk + 1, so nothing lands before it has been read.  The wait is bounded by
// `limit`; `late` comes back the same in every thread of the CTA (a block
// barrier ORs it), so the caller can leave the walk at once: after a time-out
// the slots may still change under the readers and nothing read from them
// may steer the walk.
__device__ __forceinline__ const float4 *cluster_exchange(Shared &sh, int &xk, int rank, float4 v, int C, uint32_t extra,
                                                          unsigned long long limit, bool &late) {
    const int p = xk & 1;
    if (threadIdx.x == 0) mbar_expect_tx(&sh.xbar[p], 16u * static_cast<uint32_t>(C) + extra);
    if (static_cast<int>(threadIdx.x) < C) {
        const int r = static_cast<int>(threadIdx.x);
        st_async_f4(mapa_u32(smem_u32(&sh.slot[p][rank]), r), v, mapa_u32(smem_u32(&sh.xbar[p]), r));
    }
    bool mine = false;
    const uint32_t ph = static_cast<uint32_t>(xk >> 1) & 1u;
    if (limit == 0) {
        mine = !mbar_test_wait_cluster(&sh.xbar[p], ph);   // one non-blocking test
    } else if (!mbar_try_wait_cluster(&sh.xbar[p], ph)) {
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait_cluster(&sh.xbar[p], ph)) {
            if (globaltimer() - t0 > limit) {
                mine = true;
                break;
            }
        }
    }
    late = __syncthreads_or(mine) != 0;
    ++xk;
    return sh.slot[p];
}

__device__ __forceinline__ bool nonfinite(float f) { return (f != f) || f == INFINITY; }

// Bounded wait on the row-copy barrier; false after `limit` nanoseconds (at
// the first failed try when it is 0).
__device__ bool wait_rows(uint64_t *bar, uint32_t parity, unsigned long long limit) {
    if (limit == 0) return mbar_test_wait(bar, parity);   // one non-blocking test
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait_sleep(bar, parity, 100000u))
        if (globaltimer() - t0 > limit) return false;
    return true;
}

// Logits 4g .. 4g+3 of this CTA's slice as fp32 (one 8- or 16-byte shared load).
template <int ES>
__device__ __forceinline__ float4 zgroup(const unsigned char *zs, int g) {
    if constexpr (ES == 2) {
        const uint2 v = reinterpret_cast<const uint2 *>(zs)[g];
        return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u),
                           __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
    } else {
        return reinterpret_cast<const float4 *>(zs)[g];
    }
}

template <int ES>
__global__ void __launch_bounds__(kThreads, 1) tree_sampled_kernel(const __grid_constant__ Params P) {
    extern __shared__ __align__(128) unsigned char dyn[];
    __shared__ Shared sh;
    cg::cluster_group cl = cg::this_cluster();
    const int C = P.cluster;
    const int rank = static_cast<int>(cl.block_rank());
    const int b = static_cast<int>(blockIdx.x) / C;
    const int S = P.slice, V = P.V, N = P.N, D1 = P.max_depth + 1;
    const int tid = threadIdx.x;
    constexpr bool bf16 = ES == 2;
    constexpr int es = ES;
    float *ev = reinterpret_cast<float *>(dyn);               // e of this CTA's columns
    float *qv = ev + S;                                       // q of this CTA's columns
    unsigned char *zs = dyn + 8 * static_cast<size_t>(S);     // logits of this CTA's columns, as stored
    const int lo = rank * S;
    const int n = max(0, min(S, V - lo));
    // Columns n .. npad-1 are padding (logit -inf, q 0), so every pass runs
    // over whole groups of four columns without masks.  The per-node passes
    // give group g to thread g mod 512 (consecutive threads, consecutive
    // groups: conflict-free, coalesced); the final draw gives thread t the
    // contiguous groups [t*Eg, t*Eg + Eg), Eg odd so that the threads' 16-byte
    // accesses fall in different banks, and its prefix runs in column order.
    const int npad = (n + 7) & ~7;
    const int ng = npad / 4;
    const int Eg = ((ng + kThreads - 1) / kThreads) | 1;
    const int g0 = min(ng, tid * Eg), g1 = min(ng, g0 + Eg);
    const int c0 = 4 * g0, c1 = 4 * g1;
    const float4 *ev4 = reinterpret_cast<const float4 *>(ev);
    const float4 *qv4 = reinterpret_cast<const float4 *>(qv);
    const bool lead = rank == 0 && tid == 0;
    const size_t rows = static_cast<size_t>(N) + 1;
    // bulk parts of this CTA's slices (16-byte multiples); the rest by plain loads
    const uint32_t zmain = P.zbulk ? static_cast<uint32_t>((n * es) & ~15) : 0u;
    const uint32_t qmain = P.qbulk ? static_cast<uint32_t>((n * 4) & ~15) : 0u;
    int xk = 0;          // cluster exchanges so far
    uint32_t phase = 0;
    bool bad = false, late = false;

    for (int i = tid; i < N; i += kThreads) {
        sh.tok[i] = __ldg(P.tokens + static_cast<size_t>(b) * N + i);
        sh.ua[i] = __ldg(P.u_accept + static_cast<size_t>(b) * N + i);
    }
    if (tid == 0) {
        mbar_init(&sh.bar, 1);
        mbar_init(&sh.xbar[0], 1);
        mbar_init(&sh.xbar[1], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async();
    }
    float T = __ldg(P.temperature + b);
    if (!(T > 0.0f) || T == INFINITY) {
        if (lead && P.status) atomicOr(P.status, SPEC_STATUS_BAD_TEMPERATURE);
        T = 1.0f;
    }
    const float c2 = kLog2e / T;
    if (lead) P.out_path[static_cast<size_t>(b) * D1] = 0;
    cl.sync();  // every CTA's barriers exist before anyone pushes into them

    int cur = 0, d = 0;
    for (;;) {
        const size_t roff = (static_cast<size_t>(b) * rows + cur) * static_cast<size_t>(V);
        const int kb = P.child_off[cur], m = P.child_off[cur + 1] - kb;
        // (1) this node's rows: logits always, q when it has children; the
        // children's q(x) gathered while the copies run
        const uint32_t qbytes = m > 0 ? qmain : 0u;
        if (tid == 0 && zmain + qbytes > 0) {
            fence_proxy_async();  // earlier reads of zs / qv come before the async writes
            mbar_expect_tx(&sh.bar, zmain + qbytes);
            if (zmain)
                bulk_g2s(zs, static_cast<const unsigned char *>(P.logits) + (roff + lo) * es, zmain, &sh.bar);
            if (qbytes) bulk_g2s(qv, P.q + roff + lo, qbytes, &sh.bar);
        }
        if (bf16) {
            const uint16_t *src = static_cast<const uint16_t *>(P.logits) + roff + lo;
            for (int i = static_cast<int>(zmain / 2) + tid; i < n; i += kThreads)
                reinterpret_cast<uint16_t *>(zs)[i] = __ldg(src + i);
        } else {
            const float *src = static_cast<const float *>(P.logits) + roff + lo;
            for (int i = static_cast<int>(zmain / 4) + tid; i < n; i += kThreads)
                reinterpret_cast<float *>(zs)[i] = __ldg(src + i);
        }
        if (m > 0)
            for (int i = static_cast<int>(qmain / 4) + tid; i < n; i += kThreads) qv[i] = __ldg(P.q + roff + lo + i);
        for (int i = n + tid; i < npad; i += kThreads) {
            if constexpr (bf16)
                reinterpret_cast<uint16_t *>(zs)[i] = 0xff80u;  // bf16 -inf
            else
                reinterpret_cast<float *>(zs)[i] = -INFINITY;
            qv[i] = 0.0f;
        }
        for (int k = tid; k < m; k += kThreads) {
            const int x = sh.tok[P.child_list[kb + k] - 1];
            sh.qx[k] = (x >= 0 && x < V) ? __ldg(P.q + roff + x) : 0.0f;
        }
        bool copy_late = false;
        if (zmain + qbytes > 0) {
            copy_late = !wait_rows(&sh.bar, phase, P.wait_ns);
            phase ^= 1u;
        }
        // a copy that outlived its wait ends the walk (the same in every thread)
        late = __syncthreads_or(copy_late) != 0;
        if (late) break;

        // (2) this CTA's max m_r, e = 2^((z - m_r) c2) and its sum; one cluster
        // exchange gives M = max m_r, the scales f_r = 2^((m_r - M) c2) and
        // S = sum_r f_r * sum_r, so p = e * f_r / S on rank r
        float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
        bool nan = false;
        for (int g = tid; g < ng; g += kThreads) {
            const float4 z = zgroup<ES>(zs, g);
            mx0 = fmaxf(mx0, z.x);
            mx1 = fmaxf(mx1, z.y);
            mx2 = fmaxf(mx2, z.z);
            mx3 = fmaxf(mx3, z.w);
            nan |= (z.x != z.x) | (z.y != z.y) | (z.z != z.z) | (z.w != z.w);
        }
        const float mt = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
        bad |= nan | (mt == INFINITY);
        const float mr = block_max(mt, sh);
        const float mrs = mr == -INFINITY ? 0.0f : mr;  // an empty or all -inf slice contributes nothing
        // the owner of each child's column pushes e(x) = 2^((z_x - m_r) c2) into
        // every CTA, completing on the barrier of the exchange below
        for (int k = tid; k < m; k += kThreads) {
            const int x = sh.tok[P.child_list[kb + k] - 1];
            if (x >= lo && x < lo + n) {
                const int xl = x - lo;
                float z;
                if constexpr (bf16)
                    z = __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t *>(zs)[xl]) << 16);
                else
                    z = reinterpret_cast<const float *>(zs)[xl];
                const float v = ex2((z - mrs) * c2);
                const uint32_t dl = smem_u32(&sh.exb[d & 1][k]), bl = smem_u32(&sh.xbar[xk & 1]);
                for (int r = 0; r < C; ++r) st_async_f1(mapa_u32(dl, r), v, mapa_u32(bl, r));
            }
        }
        // A thread's four running sums each take about ten terms (plain fp32,
        // relative error near 1e-7); they and everything beyond the thread
        // combine as two-float.
        float sh0, sl0;
        {
            float s0 = 0.0f, s1 = 0.0f, s2 = 0.0f, s3 = 0.0f;
            for (int g = tid; g < ng; g += kThreads) {
                const float4 z = zgroup<ES>(zs, g);
                float4 e;
                e.x = ex2((z.x - mrs) * c2);
                e.y = ex2((z.y - mrs) * c2);
                e.z = ex2((z.z - mrs) * c2);
                e.w = ex2((z.w - mrs) * c2);
                reinterpret_cast<float4 *>(ev)[g] = e;
                s0 += e.x;
                s1 += e.y;
                s2 += e.z;
                s3 += e.w;
            }
            sh0 = s0;
            sl0 = 0.0f;
            tf_add(sh0, sl0, s1, 0.0f);
            tf_add(sh0, sl0, s2, 0.0f);
            tf_add(sh0, sl0, s3, 0.0f);
        }
        block_sum2(sh0, sl0, sh);
        uint32_t nin = 0;  // children with a column: each CTA receives one 4-byte push for each
        for (int k = 0; k < m; ++k) {
            const int x = sh.tok[P.child_list[kb + k] - 1];
            nin += (x >= 0 && x < V) ? 1u : 0u;
        }
        const float4 *row =
            cluster_exchange(sh, xk, rank, make_float4(mr, sh0, sl0, 0.0f), C, 4u * nin, P.wait_ns, late);
        if (late) break;
        float M = -INFINITY;
        for (int r = 0; r < C; ++r) M = fmaxf(M, row[r].x);
        float Sh = 0.0f, Sl = 0.0f, fmine = 0.0f;
        for (int r = 0; r < C; ++r) {
            const float f = row[r].x == -INFINITY ? 0.0f : ex2((row[r].x - M) * c2);
            if (r == rank) fmine = f;
            if (tid == 0) sh.fr[r] = f;  // read only by thread 0, in the tests (the slots get reused)
            float ph, pl;
            tf_mul(row[r].y, row[r].z, f, ph, pl);
            tf_add(Sh, Sl, ph, pl);
        }
        if (!(Sh > 0.0f) || !(Sh < INFINITY)) {
            bad = true;
            Sh = 1.0f;
            Sl = 0.0f;
        }
        const float pscale = fmine / Sh;  // p = e * pscale on this rank
        // (4) children in index order; p' is max(0, p - Tm q) / ST.  Child x is
        // accepted iff q(x) == 0 or u * ST * q(x) < p(x) - Tm * q(x), both
        // sides multiplied through by S > 0 (no division)
        float Tmh = 0.0f, Tml = 0.0f, STh = 1.0f, STl = 0.0f;
        int next = -1;
        for (int k = 0; k < m; ++k) {
            if (tid == 0) {
                const int nd = P.child_list[kb + k];
                const int x = sh.tok[nd - 1];
                int acc = 0;
                if (x < 0 || x >= V) {
                    if (rank == 0 && P.status) atomicOr(P.status, SPEC_STATUS_TOKEN_RANGE);
                } else {
                    const float qx = sh.qx[k];
                    if (qx == 0.0f) {
                        acc = 1;
                    } else {
                        // e(x) * f_owner = p(x) * S
                        const float fo = sh.fr[x / S];
                        const float qS = qx * Sh;
                        const float lhs = sh.ua[nd - 1] * (STh * qS);
                        const float rhs = fmaf(-Tmh, qS, sh.exb[d & 1][k] * fo);
                        acc = lhs < rhs;
                    }
                }
                sh.dec = acc;
            }
            __syncthreads();
            if (sh.dec) {  // uniform: every thread read it after the barrier
                next = P.child_list[kb + k];
                break;
            }
            // rejected: Tm <- Tm + ST and ST <- the new residual's mass
            float Tnh = Tmh, Tnl = Tml;
            tf_add(Tnh, Tnl, STh, STl);
            const float Tnf = Tnh;
            float rh, rl;
            {
                float s0 = 0.0f, s1 = 0.0f, s2 = 0.0f, s3 = 0.0f;
                for (int g = tid; g < ng; g += kThreads) {
                    const float4 e = ev4[g], q = qv4[g];
                    s0 += fmaxf(0.0f, fmaf(-Tnf, q.x, e.x * pscale));
                    s1 += fmaxf(0.0f, fmaf(-Tnf, q.y, e.y * pscale));
                    s2 += fmaxf(0.0f, fmaf(-Tnf, q.z, e.z * pscale));
                    s3 += fmaxf(0.0f, fmaf(-Tnf, q.w, e.w * pscale));
                }
                rh = s0;
                rl = 0.0f;
                tf_add(rh, rl, s1, 0.0f);
                tf_add(rh, rl, s2, 0.0f);
                tf_add(rh, rl, s3, 0.0f);
            }
            block_sum2(rh, rl, sh);
            const float4 *rrow =
                cluster_exchange(sh, xk, rank, make_float4(rh, rl, 0.0f, 0.0f), C, 0u, P.wait_ns, late);
            if (late) break;
            float Snh = 0.0f, Snl = 0.0f;
            for (int r = 0; r < C; ++r) tf_add(Snh, Snl, rrow[r].x, rrow[r].y);
            if (Snh > 0.0f) {  // a residual of no mass leaves p' as it is
                Tmh = Tnh;
                Tml = Tnl;
                STh = Snh;
                STl = Snl;
            }
        }
        if (late) break;
        if (next < 0) {
            // one draw from p' (p, or max(0, p - Tm q) after a rejection): the
            // smallest column whose prefix exceeds t = u * total.  Prefixes run
            // over CTAs in rank order, threads in thread order and columns in
            // index order.  Every CTA finds the same CTA r* holding t from the
            // exchanged totals; in r* the thread whose chunk holds t rescans it.
            const bool resid = Tmh > 0.0f;
            const float Tf = Tmh;
            float s = 0.0f, k = 0.0f;
            int lastpos = -1;
            for (int g = g0; g < g1; ++g) {
                const float4 e = ev4[g];
                const float4 q = resid ? qv4[g] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                const float w[4] = {fmaxf(0.0f, fmaf(-Tf, q.x, e.x * pscale)), fmaxf(0.0f, fmaf(-Tf, q.y, e.y * pscale)),
                                    fmaxf(0.0f, fmaf(-Tf, q.z, e.z * pscale)), fmaxf(0.0f, fmaf(-Tf, q.w, e.w * pscale))};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    kadd(s, k, w[j]);
                    if (w[j] > 0.0f) lastpos = lo + 4 * g + j;
                }
            }
            float exh, exl, inh, inl, th, tl;
            block_scan2(s, -k, exh, exl, inh, inl, th, tl, sh);
            const int clast = block_imax(lastpos, sh);
            const float4 *trow = cluster_exchange(sh, xk, rank, make_float4(th, tl, __int_as_float(clast), 0.0f), C,
                                                  0u, P.wait_ns, late);
            if (late) break;
            // t = u * total, then the first CTA whose running end exceeds t
            float toth = 0.0f, totl = 0.0f;
            for (int r = 0; r < C; ++r) tf_add(toth, totl, trow[r].x, trow[r].y);
            const float u = __ldg(P.u_sample + static_cast<size_t>(b) * rows + cur);
            float tth, ttl;
            tf_mul(toth, totl, u, tth, ttl);
            float ch = 0.0f, cl_ = 0.0f;  // running CTA prefix
            int rstar = -1, rlast = -1;
            float bh = 0.0f, bl = 0.0f;   // prefix before r*
            for (int r = 0; r < C; ++r) {
                if (__float_as_int(trow[r].z) >= 0) rlast = r;
                float eh = ch, el = cl_;
                tf_add(eh, el, trow[r].x, trow[r].y);
                if (rstar < 0 && ((eh - tth) + (el - ttl)) > 0.0f) {
                    rstar = r;
                    bh = ch;
                    bl = cl_;
                }
                ch = eh;
                cl_ = el;
            }
            if (rstar < 0) rstar = rlast;  // t at or past the total after rounding: the last positive column
            if (rank == rstar) {
                if (tid == 0) sh.pick = -1;
                __syncthreads();
                // t relative to this CTA's first column (clamped at 0)
                float trh = tth, trl = ttl;
                tf_add(trh, trl, -bh, -bl);
                if (trh < 0.0f) trh = trl = 0.0f;
                const bool holds = c1 > c0 && ((exh - trh) + (exl - trl)) <= 0.0f && ((inh - trh) + (inl - trl)) > 0.0f;
                if (holds) {
                    float s2 = 0.0f, k2 = 0.0f;
                    int cand = -1;
                    bool done = false;
                    for (int g = g0; g < g1 && !done; ++g) {
                        const float4 e = ev4[g];
                        const float4 q = resid ? qv4[g] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                        const float w[4] = {fmaxf(0.0f, fmaf(-Tf, q.x, e.x * pscale)),
                                            fmaxf(0.0f, fmaf(-Tf, q.y, e.y * pscale)),
                                            fmaxf(0.0f, fmaf(-Tf, q.z, e.z * pscale)),
                                            fmaxf(0.0f, fmaf(-Tf, q.w, e.w * pscale))};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            if (done) continue;
                            kadd(s2, k2, w[j]);
                            if (w[j] > 0.0f) {
                                cand = lo + 4 * g + j;  // the last positive column so far: the answer if t is never passed
                                float ph = exh, pl = exl;
                                tf_add(ph, pl, s2, -k2);
                                if (((ph - trh) + (pl - trl)) > 0.0f) done = true;
                            }
                        }
                    }
                    sh.pick = cand;
                }
                __syncthreads();
                if (tid == 0) {
                    int pick = sh.pick;
                    if (pick < 0) pick = __float_as_int(trow[rank].z);  // no thread holds t: this CTA's last positive
                    if (pick < 0) pick = V - 1;
                    P.out_tokens[static_cast<size_t>(b) * D1 + d] = pick;
                }
            }
            if (lead) {
                int32_t *ot = P.out_tokens + static_cast<size_t>(b) * D1;
                int32_t *op = P.out_path + static_cast<size_t>(b) * D1;
                for (int i = d + 1; i < D1; ++i) {
                    ot[i] = -1;
                    op[i] = -1;
                }
                P.out_len[b] = d + 1;
                if (rstar < 0) ot[d] = V - 1;  // nothing positive anywhere (a non-finite row)
            }
            break;
        }
        if (lead) {
            P.out_tokens[static_cast<size_t>(b) * D1 + d] = sh.tok[next - 1];
            P.out_path[static_cast<size_t>(b) * D1 + d + 1] = next;
        }
        ++d;
        cur = next;
        __syncthreads();  // this node's reads of zs, qv and the child arrays end before the next copies
    }
    if (late) {
        // a row copy or an exchange outlived its wait: one more bounded wait
        // for the last row copy, so no copy lands here after exit
        wait_rows(&sh.bar, phase ^ 1u, kWaitLimitNs);
        if (tid == 0 && P.status) atomicOr(P.status, SPEC_STATUS_WAIT_TIMEOUT);
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
        const void *ks[2] = {reinterpret_cast<const void *>(ts::tree_sampled_kernel<2>),
                             reinterpret_cast<const void *>(ts::tree_sampled_kernel<4>)};
        for (int i = 0; i < 2 && e == cudaSuccess; ++i) {
            e = cudaFuncSetAttribute(ks[i], cudaFuncAttributeMaxDynamicSharedMemorySize, ts::kSmemBudget);
            if (e == cudaSuccess) e = cudaFuncSetAttribute(ks[i], cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        }
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
    clear_error();
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
    const int es = dtype == SPEC_BF16 ? 2 : 4;
    const int cap = ts::slice_cap(es);
    // fewest CTAs whose slices fit: a cluster per request must be resident
    // at once, and small clusters pack the GPCs best
    int C = (V + cap - 1) / cap;
    if (C < 1) C = 1;
    if (C > ts::kMaxCluster) C = ts::kMaxCluster;
    int S = round8((V + C - 1) / C);
    while (S > cap && C < ts::kMaxCluster) S = round8((V + ++C - 1) / C);
    if (S > cap) {
        char buf[96];
        snprintf(buf, sizeof buf, " (at most %d for this dtype: 16 CTAs x %d columns)", ts::kMaxCluster * cap, cap);
        return fail(SPEC_ERR_INVALID_ARG, "V is too large%s", buf);
    }
    spec_status_t st = ts_setup();
    if (st != SPEC_OK) return st;
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
    P.zbulk = (static_cast<long long>(V) * es) % 16 == 0;
    P.qbulk = V % 4 == 0;
    P.wait_ns = wait_limit_ns();
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(static_cast<unsigned>(B) * static_cast<unsigned>(C));
    cfg.blockDim = dim3(ts::kThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(S) * static_cast<size_t>(8 + es);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(C);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = P.bf16 ? cudaLaunchKernelEx(&cfg, ts::tree_sampled_kernel<2>, P)
                           : cudaLaunchKernelEx(&cfg, ts::tree_sampled_kernel<4>, P);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "sampled tree launch: %s", cudaGetErrorString(e));
    return SPEC_OK;
}
