// chain_cluster.cu -- chain verification with one thread-block cluster per
// request, for batches whose clusters all fit on the GPU at once.
//
// What it computes is the chain step of the persistent verify kernel
// (EAGLE-3 review, "Speculative Decoding": drafts checked front to back, the
// first rejection ends the step and is resampled, a bonus token when every
// draft passes; the review's small-draft section: greedy accepts iff the draft
// is the target argmax, else emits the argmax; sampling accepts x with
// probability min(1, p(x)/q(x)) and resamples from norm(max(0, p - q))).
//
// Layout.  Request b owns a cluster of C CTAs; CTA r holds columns
// [r * S, r * S + S) of a row in a ring of shared-memory stages (three).  Of
// the sixteen warps, fifteen stream rows and the last one controls the walk.
//   (1) Copies.  The control warp's lane 0 issues one bulk-async copy per row
//       slice: row 0 alone first (rows issued together land together, and
//       row 0 decides most requests), rows 1 and 2 once row 0 has landed, and
//       row j + 3 only once draft j is accepted, so no row more than two past
//       the first rejection is read.
//   (2) Streaming warps take the rows in order as they land.  Each thread
//       folds the 8-column groups stid, stid + 480, ... of the row into
//       running statistics (the bonus row k: a contiguous chunk of groups
//       per thread, the layout its draw scans), each warp leaves one partial
//       per row and frees the stage; nothing waits on a block reduction.
//         * greedy (T == 0): the slice's maximum and the first column holding it;
//           the row's argmax is the largest value, lowest column.
//         * sampled: the slice's max m_r and sum_r = sum 2^((z - m_r) log2e/T)
//           (two-float), and e(x) on its own scale in the CTA holding the draft
//           token's column.  M = max m_r, S = sum_r 2^((m_r - M) log2e/T) sum_r,
//           and the accept test u q(x) S < e(x) 2^((m_owner - M) log2e/T)
//           needs no division.
//   (3) The control warp, row by row: the warps' partials become the CTA's
//       statistics of the row, one exchange sends them to every CTA of the
//       cluster (st.async into a slot of each CTA, completing on the
//       receiver's mbarrier), and every CTA takes draft j's decision from the
//       same C values.
//   (4) The first rejection a (or k) ends the walk.  A greedy request emits
//       the argmax of row a; a sampled one draws by inverse CDF over the
//       residual max(0, p - q) of row a (p of row k for the bonus token; p when
//       the residual has no mass): per-thread sums over contiguous chunks of
//       groups, a block scan, one exchange of the CTA totals, then one warp
//       rescans the chunk holding t = u * total, a lane per group.  Row a's
//       logits are still in their stage; q of row a is copied into the other
//       two stages once the rows in flight there have landed.  The bonus row
//       needs no pass of its own: its streaming fold already holds each
//       chunk's sum.
//
// Every wait is bounded (the caller's limit); a wait that runs out ends the
// walk for the whole CTA (a block barrier ORs the outcome) and sets
// SPEC_STATUS_WAIT_TIMEOUT; copies in flight are waited for before exit and
// no CTA leaves before the cluster barrier, so no remote store lands in a
// finished CTA.
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <climits>
#include <mutex>
#include <utility>
#include <vector>

#include "common.h"
#include "ptx.cuh"
#include "spec_verify.h"
#include "twofloat.cuh"

namespace cg = cooperative_groups;

namespace sv {
namespace cc {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kCtrlWarp = kWarps - 1;          // decisions and copies; the other warps stream the rows
constexpr int kStreamWarps = kWarps - 1;
constexpr int kStreamThreads = kStreamWarps * 32;
constexpr int kMaxCluster = 16;
constexpr int kSmemBudget = 212 * 1024;   // dynamic: the ring, or the drawn row's slices
constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned long long kWaitLimitNs = 500000000ull;   // the limit on copies in flight at exit

struct Params {
    const void *logits;          // [B, k+1, V] bf16 bits or fp32
    const float *q;              // [B, k, V] or null (every request greedy)
    const int32_t *tokens;       // [B, k]
    const float *temperature;    // [B] or null
    const float *u_accept;       // [B, k] or null
    const float *u_sample;       // [B, k+1] or null
    int32_t *out_tokens;         // [B, k+1]
    int32_t *out_count;          // [B]
    int64_t *slots;              // [B, k+1] or null: slot_mapping fix-up
    int64_t pad;
    int32_t *status;             // one word or null
    unsigned long long *stats;   // workspace diagnostic counters or null
    unsigned long long logits_end, q_end;
    unsigned long long wait_ns;
    int B, k, V, C, S;           // requests, drafts, vocabulary, CTAs per request, columns per CTA
    int zbulk, qbulk;            // rows start on 16-byte boundaries: bulk copies allowed
    int stages;                  // ring stages
    unsigned long long stage_bytes;
    unsigned long long smem;     // dynamic shared memory of the launch
};

constexpr int kMaxRowsCC = 16;   // rows per request (k + 1) this kernel takes
constexpr int kMaxStages = 3;    // the ring

struct Shared {
    uint64_t bar;                      // the drawn row's q copies
    uint64_t full[kMaxStages];         // ring stage holds its row
    uint64_t empty[kMaxStages];        // every streaming warp is done with the stage's row
    uint64_t rbar[kMaxRowsCC];         // every rank's statistics of row i arrived
    uint64_t xbar[2];                  // draw exchanges, by parity
    float4 slot[2][kMaxCluster];       // pushed by every rank
    float4 rows[kMaxCluster][kMaxRowsCC];   // every rank's statistics of every row
    float4 mine[kMaxRowsCC];           // this CTA's statistics of every row walked
    float pa[kMaxRowsCC][kWarps];      // per-warp partials of every row: sampled (max, sum hi, sum lo),
    float pb[kMaxRowsCC][kWarps];      // greedy (value, column)
    float pc[kMaxRowsCC][kWarps];
    float zx[kMaxRowsCC];              // the draft token's logit, in the CTA holding its column
    float rowM[kMaxRowsCC];            // sampled: row max M
    tf rowS[kMaxRowsCC];               // ... and sum S (two-float)
    int arg[kMaxRowsCC];               // greedy: row argmax
    int acc[kMaxRowsCC];               // draft i passes its test
    float ws[kWarps], wc[kWarps], wxs[kWarps], wxc[kWarps];
    int end_row;                       // the walk's last row, once decided (rows past it are skipped)
    int abort;                         // a wait of the walk ran out
    int qfail;                         // a wait before the q copies ran out
    int a;                             // the first rejection (k: every draft accepted)
    int issued;                        // rows copied into the ring
    int wi[kWarps];
    float tot[2];
    int holder;                        // the thread whose chunk holds the draw point
    tf hex;                            // its exclusive prefix
    int32_t tok[kMaxRowsCC];           // the request's draft tokens
    float ua[kMaxRowsCC];              // its accept uniforms
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Bounded wait of one thread on a barrier that remote CTAs complete.
__device__ __forceinline__ bool cluster_bar_wait(uint64_t *bar, uint32_t ph, unsigned long long limit) {
    if (limit == 0) return mbar_test_wait_cluster(bar, ph);
    if (mbar_try_wait_cluster(bar, ph)) return true;
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait_cluster(bar, ph))
        if (globaltimer() - t0 > limit) return false;
    return true;
}

__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Eight logits of group g (8 columns) of the slice, as fp32.
template <int ES>
__device__ __forceinline__ void group8(const unsigned char *zs, int g, float x[8]) {
    if constexpr (ES == 2) {
        const uint4 w = reinterpret_cast<const uint4 *>(zs)[g];
        x[0] = bf_lo(w.x); x[1] = bf_hi(w.x); x[2] = bf_lo(w.y); x[3] = bf_hi(w.y);
        x[4] = bf_lo(w.z); x[5] = bf_hi(w.z); x[6] = bf_lo(w.w); x[7] = bf_hi(w.w);
    } else {
        const float4 a = reinterpret_cast<const float4 *>(zs)[2 * g], c = reinterpret_cast<const float4 *>(zs)[2 * g + 1];
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = c.x; x[5] = c.y; x[6] = c.z; x[7] = c.w;
    }
}

// Eight logits of group g read from global memory (row slice base zg, n
// columns; -inf past the end): the groups a bulk copy does not cover.
template <int ES>
__device__ __forceinline__ void group8_global(const void *zg, int g, int n, float x[8]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int c = 8 * g + j;
        if (c >= n)
            x[j] = -INFINITY;
        else if constexpr (ES == 2)
            x[j] = __uint_as_float(static_cast<uint32_t>(__ldg(static_cast<const uint16_t *>(zg) + c)) << 16);
        else
            x[j] = __ldg(static_cast<const float *>(zg) + c);
    }
}

// Bounded wait on a cluster-scope barrier phase; `late` comes back the same in
// every thread of the CTA.
__device__ __forceinline__ bool cluster_phase_late(uint64_t *bar, uint32_t ph, unsigned long long limit) {
    bool mine = false;
    if (limit == 0) {
        mine = !mbar_test_wait_cluster(bar, ph);
    } else if (!mbar_try_wait_cluster(bar, ph)) {
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait_cluster(bar, ph)) {
            if (globaltimer() - t0 > limit) {
                mine = true;
                break;
            }
        }
    }
    return __syncthreads_or(mine) != 0;
}

// Exchange number xk of the draw (see the file comment).
__device__ __forceinline__ const float4 *exchange(Shared &sh, int &xk, int rank, float4 v, int C,
                                                  unsigned long long limit, bool &late) {
    const int p = xk & 1;
    if (threadIdx.x == 0) mbar_expect_tx(&sh.xbar[p], 16u * static_cast<uint32_t>(C));
    if (static_cast<int>(threadIdx.x) < C) {
        const int r = static_cast<int>(threadIdx.x);
        st_async_f4(mapa_u32(smem_u32(&sh.slot[p][rank]), r), v, mapa_u32(smem_u32(&sh.xbar[p]), r));
    }
    late = cluster_phase_late(&sh.xbar[p], static_cast<uint32_t>(xk >> 1) & 1u, limit);
    ++xk;
    return sh.slot[p];
}

__device__ bool wait_copies(uint64_t *bar, uint32_t parity, unsigned long long limit) {
    if (limit == 0) return mbar_test_wait(bar, parity);
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait_sleep(bar, parity, 100000u))
        if (globaltimer() - t0 > limit) return false;
    return true;
}

// Argmax step: (ov, oi) replaces (v, i) when larger, or equal at a lower column.
__device__ __forceinline__ void argmax_take(float &v, int &i, float ov, int oi) {
    if (ov > v || (ov == v && static_cast<unsigned>(oi) < static_cast<unsigned>(i))) {
        v = ov;
        i = oi;
    }
}

// Exclusive and inclusive two-float prefixes, in thread order, of the threads'
// values, and the block total (every thread).
__device__ __forceinline__ void block_scan(tf v, tf &ex, tf &in, tf &tot, Shared &sh) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    tf is = warp_incl_scan_tf(v, lane);
    if (lane == 31) {
        sh.ws[w] = is.h;
        sh.wc[w] = is.l;
    }
    __syncthreads();
    if (w == 0) {   // warp 0 scans the warps' totals
        const tf t = lane < kWarps ? tf{sh.ws[lane], sh.wc[lane]} : tf_of(0.0f);
        const tf inc = warp_incl_scan_tf(t, lane);
        const tf up{__shfl_up_sync(0xffffffffu, inc.h, 1), __shfl_up_sync(0xffffffffu, inc.l, 1)};
        if (lane < kWarps) {
            sh.wxs[lane] = lane ? up.h : 0.0f;
            sh.wxc[lane] = lane ? up.l : 0.0f;
        }
        if (lane == kWarps - 1) {
            sh.tot[0] = inc.h;
            sh.tot[1] = inc.l;
        }
    }
    __syncthreads();
    const tf base{sh.wxs[w], sh.wxc[w]};
    in = tf_add(base, is);
    ex = tf_add(in, tf_neg(v));
    tot = tf{sh.tot[0], sh.tot[1]};
}

// The drawn row's slices in shared memory: the logits at zs, q split at group
// gh between qa (groups below gh) and qb.
template <int ES>
struct DrawRow {
    const unsigned char *zs;   // groups below gbulk; the rest from zg
    const void *zg;
    int gbulk, n;
    const float *qa, *qb;
    int gh;
    bool resid;
    float c2, nm, pscale;
    // The eight weights of group g: p (times a common factor) or max(0, p - q).
    __device__ __forceinline__ void weights(int g, float w[8]) const {
        float z[8];
        if (g < gbulk)
            group8<ES>(zs, g, z);
        else
            group8_global<ES>(zg, g, n, z);
#pragma unroll
        for (int j = 0; j < 8; ++j) w[j] = ex2(fmaf(z[j], c2, nm)) * pscale;
        if (resid) {
            const float *qs = g < gh ? qa + 8 * g : qb + 8 * (g - gh);
            const float4 q0 = reinterpret_cast<const float4 *>(qs)[0], q1 = reinterpret_cast<const float4 *>(qs)[1];
            w[0] = fmaxf(0.0f, w[0] - q0.x); w[1] = fmaxf(0.0f, w[1] - q0.y);
            w[2] = fmaxf(0.0f, w[2] - q0.z); w[3] = fmaxf(0.0f, w[3] - q0.w);
            w[4] = fmaxf(0.0f, w[4] - q1.x); w[5] = fmaxf(0.0f, w[5] - q1.y);
            w[6] = fmaxf(0.0f, w[6] - q1.z); w[7] = fmaxf(0.0f, w[7] - q1.w);
        }
    }
    __device__ __forceinline__ float gsum(const float w[8]) const {
        float s = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) s += w[j];
        return s;
    }
};

template <int ES>
__global__ void __launch_bounds__(kThreads, 1) chain_cluster_kernel(const __grid_constant__ Params P) {
    extern __shared__ __align__(128) unsigned char dyn[];
    __shared__ Shared sh;
    cg::cluster_group cl = cg::this_cluster();
    const int C = P.C;
    const int rank = static_cast<int>(cl.block_rank());
    const int b = static_cast<int>(blockIdx.x) / C;
    const int S = P.S, V = P.V, k = P.k, R = k + 1;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool ctrl = warp == kCtrlWarp;
    const int tctl = kCtrlWarp * 32;               // issues every bulk copy and owns their bookkeeping
    const int lo = rank * S;
    const int n = max(0, min(S, V - lo));          // columns of this CTA
    const int ng = (n + 7) >> 3;                   // 8-column groups (the last one padded)
    const bool lead = rank == 0 && tid == 0;
    const uint32_t zmain = P.zbulk ? static_cast<uint32_t>((n * ES) & ~15) : 0u;
    const uint32_t qmain = P.qbulk ? static_cast<uint32_t>((n * 4) & ~15) : 0u;
    const int NS = P.stages;
    const size_t stage_bytes = P.stage_bytes;
    const int gbulk = static_cast<int>(zmain / (8 * ES));   // groups wholly copied into a stage
    auto zrow = [&](int i) -> size_t { return (static_cast<size_t>(b) * R + i) * static_cast<size_t>(V); };
    auto qrow = [&](int i) -> size_t { return (static_cast<size_t>(b) * k + i) * static_cast<size_t>(V); };
    unsigned long long bytes = 0;
    // Row j into ring stage j % NS (control lane 0): one bulk copy of the
    // 16-byte aligned part of the slice; the rest by plain loads after the wait.
    // A row with nothing to copy in bulk completes its stage by a plain arrive.
    auto issue = [&](int j) {
        const int st = j % NS;
        if (zmain) {
            fence_proxy_async();
            mbar_expect_tx(&sh.full[st], zmain);
            bulk_g2s(dyn + st * stage_bytes, static_cast<const unsigned char *>(P.logits) + (zrow(j) + lo) * ES, zmain,
                     &sh.full[st]);
            bytes += zmain;
        } else {
            mbar_arrive(&sh.full[st]);
        }
    };
    const float T = P.temperature ? __ldg(P.temperature + b) : 0.0f;   // first used after the ring starts
    // The control warp holds draft i's token, accept uniform and q_i(x) in lane
    // i.  Its lane 0 starts the ring before anything waits on a load: loads
    // issued after the whole grid's first copies queue behind them.
    int xr = -1;
    float uar = 0.0f, qxr = 0.0f;
    if (ctrl) {
        if (lane == 0) {
            mbar_init(&sh.bar, 1);
            for (int i = 0; i < kMaxStages; ++i) {
                mbar_init(&sh.full[i], 1);
                mbar_init(&sh.empty[i], kStreamWarps);
            }
            for (int i = 0; i < kMaxRowsCC; ++i) mbar_init(&sh.rbar[i], 1);
            mbar_init(&sh.xbar[0], 1);
            mbar_init(&sh.xbar[1], 1);
            sh.end_row = R;
            sh.abort = 0;
            sh.qfail = 0;
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            fence_proxy_async();
            // row 0 alone first when the rows are copied in bulk: rows issued
            // together land together, and row 0 decides most requests
            for (int j = 0; j < (zmain ? 1 : min(NS, R)); ++j) issue(j);
        }
        __syncwarp();
        if (lane < k) {
            xr = __ldg(P.tokens + static_cast<size_t>(b) * k + lane);
            uar = P.u_accept ? __ldg(P.u_accept + static_cast<size_t>(b) * k + lane) : 0.0f;
            sh.tok[lane] = xr;
            if (P.q && xr >= 0 && xr < V) qxr = __ldg(P.q + qrow(lane) + xr);   // used at the decisions
        }
    }
    // this CTA's barriers exist; the other CTAs wait for that only before their
    // first push into them
    cluster_arrive();
    __syncthreads();

    const bool greedy = !(T > 0.0f) || !P.q;
    const float c2 = greedy ? 0.0f : kLog2e / T;
    int a = -1;
    int issued = min(NS, R);   // rows copied into the ring (control warp)
    bool bad = false;
    // the bonus row (row k) is folded in contiguous chunks of Es groups per
    // streaming thread, the layout its draw scans: when the walk accepts every
    // draft, each thread's fold is already its chunk's share of p
    const int Es = ((ng + kStreamThreads - 1) / kStreamThreads) | 1;   // odd: bank spread
    float bonus_m = -INFINITY, bonus_s = 0.0f;
    int bonus_last = -1;   // the chunk's last group with a logit above -inf
    if (!ctrl) {
        // (1) streaming warps: rows in order, each thread folding the groups
        // stid, stid + 480, ... of the row (the bonus row: its contiguous
        // chunk); a warp partial per row
        const int stid = tid;   // the control warp is the last one
        for (int j = 0; j < R; ++j) {
            const int st = j % NS;
            unsigned char *zr = dyn + st * stage_bytes;
            bool ok = wait_copies(&sh.full[st], static_cast<uint32_t>((j / NS) & 1), P.wait_ns);
            if (!ok) {
                atomicOr(&sh.abort, 1);
                break;
            }
            if (j > *reinterpret_cast<volatile int *>(&sh.end_row)) break;   // the chain ended before row j
            const void *zg = static_cast<const unsigned char *>(P.logits) + (zrow(j) + lo) * ES;
            if (stid == 0) {
                const int x = j < k ? sh.tok[j] : -1;
                float zx = 0.0f;
                if (x >= lo && x < lo + n) {
                    const int c = x - lo;
                    const unsigned char *src = c < 8 * gbulk ? zr : static_cast<const unsigned char *>(zg);
                    if constexpr (ES == 2)
                        zx = __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t *>(src)[c]) << 16);
                    else
                        zx = reinterpret_cast<const float *>(src)[c];
                }
                sh.zx[j] = zx;
            }
            if (greedy) {
                float v = -INFINITY;
                int gi = INT_MAX;
                bool nan = false;
                for (int g = stid; g < ng; g += kStreamThreads) {
                    float z[8];
                    if (g < gbulk)
                        group8<ES>(zr, g, z);
                    else
                        group8_global<ES>(zg, g, n, z);
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) {
                        nan |= (z[jj] != z[jj]) || z[jj] == INFINITY;
                        if (z[jj] > v) {
                            v = z[jj];
                            gi = lo + 8 * g + jj;
                        }
                    }
                }
                bad |= nan;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    argmax_take(v, gi, __shfl_xor_sync(0xffffffffu, v, o), __shfl_xor_sync(0xffffffffu, gi, o));
                if (lane == 0) {
                    sh.pa[j][warp] = v;
                    sh.pb[j][warp] = __int_as_float(gi);
                }
            } else {
                // online max m and sums s0 + s1 relative to it; a NaN or +inf
                // logit turns the sum into NaN, a -inf one adds 0
                float m = -INFINITY, nm = 0.0f, s0 = 0.0f, s1 = 0.0f;
                // one group into the running max and sums; true if it holds a logit above -inf
                auto fold = [&](int g) {
                    float z[8];
                    if (g < gbulk)
                        group8<ES>(zr, g, z);
                    else
                        group8_global<ES>(zg, g, n, z);
                    const float gm =
                        fmaxf(fmaxf(fmaxf(z[0], z[1]), fmaxf(z[2], z[3])), fmaxf(fmaxf(z[4], z[5]), fmaxf(z[6], z[7])));
                    if (gm > m) {
                        const float f = ex2((m - gm) * c2);
                        s0 *= f;
                        s1 *= f;
                        m = gm;
                        nm = -m * c2;
                    }
                    s0 += ex2(fmaf(z[0], c2, nm));
                    s1 += ex2(fmaf(z[1], c2, nm));
                    s0 += ex2(fmaf(z[2], c2, nm));
                    s1 += ex2(fmaf(z[3], c2, nm));
                    s0 += ex2(fmaf(z[4], c2, nm));
                    s1 += ex2(fmaf(z[5], c2, nm));
                    s0 += ex2(fmaf(z[6], c2, nm));
                    s1 += ex2(fmaf(z[7], c2, nm));
                    return gm > -INFINITY;
                };
                if (j == R - 1) {
                    const int g0 = min(ng, stid * Es), g1 = min(ng, g0 + Es);
                    for (int g = g0; g < g1; ++g)
                        if (fold(g)) bonus_last = g;
                } else {
                    for (int g = stid; g < ng; g += kStreamThreads) fold(g);
                }
                const float s = s0 + s1;
                if (j == R - 1) {
                    bonus_m = m;
                    bonus_s = s;
                }
                bad |= s != s;
                float wm = m;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, o));
                tf t = tf_of((m == -INFINITY || !(s == s)) ? 0.0f : s * ex2((m - wm) * c2));
                t = warp_sum_tf(t);
                if (lane == 0) {
                    sh.pa[j][warp] = wm;
                    sh.pb[j][warp] = t.h;
                    sh.pc[j][warp] = t.l;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.empty[st]);   // this warp is done with the stage (and its partial is written)
        }
    } else {
        // (2) control warp: per row, the CTA's statistics from the warps'
        // partials, one exchange with the cluster, the decision; row j + NS is
        // copied only once row j is accepted.  First the rest of the ring goes
        // out, once row 0 has landed.
        bool started = true;
        if (zmain && min(NS, R) > 1) {
            if (lane == 0) started = wait_copies(&sh.full[0], 0u, P.wait_ns);
            started = __shfl_sync(0xffffffffu, started, 0) != 0;
            if (started && lane == 0)
                for (int j = 1; j < min(NS, R); ++j) issue(j);
            if (!started) {
                issued = 1;
                if (lane == 0) atomicOr(&sh.abort, 1);
            }
        }
        cluster_wait();   // every CTA's barriers are initialised
        for (int j = 0; j < R && started; ++j) {
            const int st = j % NS;
            const bool drained = wait_copies(&sh.empty[st], static_cast<uint32_t>((j / NS) & 1), P.wait_ns);
            if (!__all_sync(0xffffffffu, drained)) {
                atomicOr(&sh.abort, 1);
                break;
            }
            const int x = __shfl_sync(0xffffffffu, xr, j & 31);
            const bool x_ok = j < k && x >= 0 && x < V;
            const int l = lane < kStreamWarps ? lane : 0;
            float4 mine;
            if (greedy) {
                float v = lane < kStreamWarps ? sh.pa[j][l] : -INFINITY;
                int gi = lane < kStreamWarps ? __float_as_int(sh.pb[j][l]) : INT_MAX;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    argmax_take(v, gi, __shfl_xor_sync(0xffffffffu, v, o), __shfl_xor_sync(0xffffffffu, gi, o));
                mine = make_float4(v, __int_as_float(gi), 0.0f, 0.0f);
            } else {
                const float wm = lane < kStreamWarps ? sh.pa[j][l] : -INFINITY;
                float bm = wm;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, o));
                tf u = tf_of(0.0f);
                if (wm != -INFINITY) u = tf_mulf(tf{sh.pb[j][l], sh.pc[j][l]}, ex2((wm - bm) * c2));
                u = warp_sum_tf(u);
                // e(x) on this CTA's scale, in the CTA holding the draft token's column
                const float ex = (x_ok && x >= lo && x < lo + n && bm != -INFINITY) ? ex2((sh.zx[j] - bm) * c2) : 0.0f;
                mine = make_float4(bm, u.h, u.l, ex);
            }
            if (lane == 0) mbar_expect_tx(&sh.rbar[j], 16u * static_cast<uint32_t>(C));
            if (lane < C)
                st_async_f4(mapa_u32(smem_u32(&sh.rows[rank][j]), lane), mine, mapa_u32(smem_u32(&sh.rbar[j]), lane));
            const bool got = cluster_bar_wait(&sh.rbar[j], 0, P.wait_ns);
            if (!__all_sync(0xffffffffu, got)) {
                atomicOr(&sh.abort, 1);
                break;
            }
            // the decision on draft j from every rank's statistics of row j
            const bool on = lane < C;
            const float4 rv = on ? sh.rows[lane][j] : make_float4(-INFINITY, __int_as_float(INT_MAX), 0.0f, 0.0f);
            bool accept = false, rbad = false;
            if (greedy) {
                float v = rv.x;
                int gi = __float_as_int(rv.y);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    argmax_take(v, gi, __shfl_xor_sync(0xffffffffu, v, o), __shfl_xor_sync(0xffffffffu, gi, o));
                rbad = !(v > -INFINITY);
                const int g = (gi >= 0 && gi < V) ? gi : 0;
                if (lane == 0) sh.arg[j] = g;
                accept = x_ok && x == g;
            } else {
                float M = rv.x;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
                const float f = (!on || rv.x == -INFINITY) ? 0.0f : ex2((rv.x - M) * c2);
                tf St = on ? tf_mulf(tf{rv.y, rv.z}, f) : tf_of(0.0f);
                St = warp_sum_tf(St);
                const int owner = x_ok ? x / S : 0;
                const float eown = __shfl_sync(0xffffffffu, rv.w * f, owner & 31);
                if (!(St.h > 0.0f) || !(St.h < INFINITY)) {
                    rbad = true;
                    St = tf_of(1.0f);
                }
                if (lane == 0) {
                    sh.rowM[j] = M;
                    sh.rowS[j] = St;
                    sh.mine[j] = mine;
                }
                const float qx = __shfl_sync(0xffffffffu, qxr, j & 31), ua = __shfl_sync(0xffffffffu, uar, j & 31);
                // u < p(x) / q(x), with p(x) = e(x) f_owner / S, multiplied through by q(x) S
                accept = x_ok && (qx == 0.0f || ua * (qx * St.h) < eown);
            }
            if (lane == 0) bad |= rbad;
            if (!accept) {
                a = j;   // the first rejection, or row k: the bonus row
                break;
            }
            if (j + NS < R) {
                if (lane == 0) issue(j + NS);
                ++issued;
            }
        }
        // a draft token outside [0, V) anywhere in the request is reported (as a
        // rejection where the walk reaches it)
        const bool bad_token = __any_sync(0xffffffffu, lane < k && (xr < 0 || xr >= V));
        if (rank == 0 && lane == 0 && bad_token && P.status) atomicOr(P.status, SPEC_STATUS_TOKEN_RANGE);
        if (lane == 0) {
            sh.a = a;
            sh.issued = issued;
            if (a >= 0) {
                // streaming warps past the end stop at the next row they wake
                // on; the first row never copied is completed by a plain arrive
                // (its stage's previous row was consumed, so that phase is done)
                *reinterpret_cast<volatile int *>(&sh.end_row) = a;
                if (issued < R) mbar_arrive(&sh.full[issued % NS]);
            }
        }
        __syncwarp();
    }
    if (!ctrl) cluster_wait();
    __syncthreads();
    bool late = sh.abort != 0;
    a = late ? -1 : sh.a;
    late |= a < 0;
    const int fake_stage = (!late && sh.issued < R) ? sh.issued % NS : -1;   // its last phase was the plain arrive
    const int token = (!late && greedy) ? sh.arg[a] : 0;

    int xk = 0;
    bool drawn_copy = false;   // the drawn row's q copies were issued
    if (!late && !greedy) {
        // (3) inverse-CDF draw over the residual max(0, p - q) of row a (p when
        // a == k, or when the residual has no mass); p = e 2^((m_r - M) c2) / S.
        // Row a's logits are still in stage a % NS; q of row a goes into the
        // other stages once the rows copied past the rejection have landed.
        const bool want_q = a < k;
        const int sa = a % NS;
        const int o1 = sa == 0 ? 1 : 0, o2 = sa == 2 ? 1 : 2;   // the other two stages, in order
        const int gh = ES == 2 ? (ng + 1) >> 1 : ng;             // groups of q in the first of them
        const unsigned char *zs = dyn + static_cast<size_t>(sa) * stage_bytes;
        float *qa = reinterpret_cast<float *>(dyn + static_cast<size_t>(o1) * stage_bytes);
        float *qb = reinterpret_cast<float *>(dyn + static_cast<size_t>(o2) * stage_bytes);
        auto qdst = [&](int c) -> float * { return c < 8 * gh ? qa + c : qb + (c - 8 * gh); };
        uint32_t qa_bytes = 0, qb_bytes = 0;
        if (want_q && qmain) {
            const uint32_t cut = static_cast<uint32_t>(gh) * 32u;
            qa_bytes = qmain < cut ? qmain : cut;
            qb_bytes = qmain - qa_bytes;
        }
        if (want_q) {
            if (tid == tctl) {
                // the last row copied into stage s past the rejection (still in flight), or -1
                auto last_row = [&](int s) {
                    int r = -1;
                    for (int j = a + 1; j < issued; ++j)
                        if (j % NS == s) r = j;
                    return r;
                };
                bool ok = true;
                const int r1 = last_row(o1);
                if (r1 >= 0) ok = wait_copies(&sh.full[o1], static_cast<uint32_t>((r1 / NS) & 1), P.wait_ns);
                if (ok && qa_bytes) {
                    mbar_expect_tx_only(&sh.bar, qa_bytes);
                    fence_proxy_async();
                    bulk_g2s(qa, P.q + qrow(a) + lo, qa_bytes, &sh.bar);
                    bytes += qa_bytes;
                }
                if (gh < ng) {
                    const int r2 = last_row(o2);
                    if (ok && r2 >= 0) ok = wait_copies(&sh.full[o2], static_cast<uint32_t>((r2 / NS) & 1), P.wait_ns);
                    if (ok && qb_bytes) {
                        mbar_expect_tx_only(&sh.bar, qb_bytes);
                        fence_proxy_async();
                        bulk_g2s(qb, P.q + qrow(a) + lo + 8 * gh, qb_bytes, &sh.bar);
                        bytes += qb_bytes;
                    }
                }
                mbar_arrive(&sh.bar);   // the phase ends when the copies issued above have landed
                sh.qfail = ok ? 0 : 1;
            }
            drawn_copy = true;
            __syncthreads();
            if (!sh.qfail) {
                // plain loads of what the bulk copies leave, and the padding
                for (int c = static_cast<int>((qa_bytes + qb_bytes) / 4) + tid; c < n; c += kThreads)
                    *qdst(c) = __ldg(P.q + qrow(a) + lo + c);
                for (int c = n + tid; c < 8 * ng; c += kThreads) *qdst(c) = 0.0f;
            }
            const bool copy_late = sh.qfail || !wait_copies(&sh.bar, 0, P.wait_ns);
            late = __syncthreads_or(copy_late) != 0;
        }

        const float u = P.u_sample ? __ldg(P.u_sample + static_cast<size_t>(b) * R + a) : 0.0f;
        const float mr = sh.mine[a].x, M = sh.rowM[a];
        const float Sh = sh.rowS[a].h;
        DrawRow<ES> D;
        D.zs = zs;
        D.zg = static_cast<const unsigned char *>(P.logits) + (zrow(a) + lo) * ES;
        D.gbulk = gbulk;
        D.n = n;
        D.qa = qa;
        D.qb = qb;
        D.gh = gh;
        D.resid = want_q;
        D.c2 = c2;
        D.nm = mr == -INFINITY ? 0.0f : -mr * c2;
        D.pscale = (mr == -INFINITY ? 0.0f : ex2((mr - M) * c2)) / Sh;
        // contiguous chunks of groups per thread (odd length: bank spread); the
        // bonus row keeps the chunks its streaming pass folded
        const bool bonus = a == R - 1;
        const int Eg = bonus ? Es : (((ng + kThreads - 1) / kThreads) | 1);
        const int g0 = min(ng, tid * Eg), g1 = min(ng, g0 + Eg);
        for (int attempt = 0; attempt < 2 && !late; ++attempt) {
            if (tid == 0) sh.holder = INT_MAX;
            tf th = tf_of(0.0f);
            int lastg = -1;
            if (bonus) {
                // the streaming pass's fold of this chunk, rescaled to the draw's
                // units: sum over the chunk of 2^((z - m_t) c2), times
                // 2^((m_t - m_r) c2) pscale
                if (mr != -INFINITY && bonus_m != -INFINITY)
                    th = tf_of(bonus_s * (ex2((bonus_m - mr) * c2) * D.pscale));
                lastg = bonus_last;
            } else if (mr != -INFINITY)
                for (int g = g0; g < g1; ++g) {
                    float w[8];
                    D.weights(g, w);
                    const float ws = D.gsum(w);
                    if (ws > 0.0f) lastg = g;
                    th = tf_add(th, tf_of(ws));
                }
            tf ex, in, tot;
            block_scan(th, ex, in, tot, sh);
            int clast = lastg;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) clast = max(clast, __shfl_xor_sync(0xffffffffu, clast, o));
            if (lane == 0) sh.wi[warp] = clast;
            __syncthreads();
            clast = sh.wi[0];
            for (int w = 1; w < kWarps; ++w) clast = max(clast, sh.wi[w]);
            const float4 *trow = exchange(sh, xk, rank, make_float4(tot.h, tot.l, __int_as_float(clast), 0.0f),
                                          C, P.wait_ns, late);
            if (late) break;
            // every warp scans the CTA totals in rank order (lane r: rank r)
            const tf own_r = lane < C ? tf{trow[lane].x, trow[lane].y} : tf_of(0.0f);
            const tf end_r = warp_incl_scan_tf(own_r, lane);
            const tf Z = tf_shfl(end_r, C - 1);
            if (D.resid && !(Z.h > 0.0f)) {
                D.resid = false;   // a residual of no mass: sample from p
                __syncthreads();
                continue;
            }
            const tf t = tf_mulf(Z, u);
            // the CTA holding t: the first whose running end exceeds t
            const unsigned past = __ballot_sync(0xffffffffu, lane < C && tf_gt(end_r, t));
            const unsigned pos = __ballot_sync(0xffffffffu, lane < C && __float_as_int(trow[lane].z) >= 0);
            // t at or past the total after rounding: the last CTA with a positive column
            const int rstar = past ? __ffs(past) - 1 : (pos ? 31 - __clz(pos) : -1);
            const tf up{__shfl_up_sync(0xffffffffu, end_r.h, 1), __shfl_up_sync(0xffffffffu, end_r.l, 1)};
            const int rs = rstar > 0 ? rstar : 0;
            tf before = tf{__shfl_sync(0xffffffffu, up.h, rs), __shfl_sync(0xffffffffu, up.l, rs)};
            if (rstar <= 0) before = tf_of(0.0f);
            if (rank == rstar) {
                tf tr = tf_add(t, tf_neg(before));   // t relative to this CTA's first column
                if (tr.h < 0.0f) tr = tf_of(0.0f);
                if (g1 > g0 && !tf_gt(ex, tr) && tf_gt(in, tr)) atomicMin(&sh.holder, tid);
                __syncthreads();
                if (tid == sh.holder) sh.hex = ex;
                __syncthreads();
                if (warp == 0) {
                    const int h = sh.holder;
                    int pick = -1;
                    if (h != INT_MAX) {
                        // the holder's chunk, 32 groups at a time: a lane per
                        // group, a scan of the group sums, then the crossing
                        // group's columns in order
                        const int hg0 = h * Eg, hg1 = min(ng, hg0 + Eg);
                        tf acc0 = sh.hex;
                        int lastcol = -1;
                        for (int base = hg0; base < hg1 && pick < 0; base += 32) {
                            const int g = base + lane;
                            float w[8];
                            float gs = 0.0f;
                            if (g < hg1) {
                                D.weights(g, w);
                                gs = D.gsum(w);
                            } else {
#pragma unroll
                                for (int jj = 0; jj < 8; ++jj) w[jj] = 0.0f;
                            }
                            const tf own = tf_of(gs);
                            const tf endl = tf_add(acc0, warp_incl_scan_tf(own, lane));
                            const unsigned cross = __ballot_sync(0xffffffffu, g < hg1 && tf_gt(endl, tr));
                            int mine_pick = -1;
                            if (cross) {
                                const int L = __ffs(cross) - 1;
                                if (lane == L) {
                                    tf acc = tf_add(endl, tf_neg(own));   // the running sum before group g
                                    bool done = false;
#pragma unroll
                                    for (int jj = 0; jj < 8; ++jj)
                                        if (!done && w[jj] > 0.0f) {
                                            mine_pick = lo + 8 * g + jj;
                                            acc = tf_add(acc, tf_of(w[jj]));
                                            done = tf_gt(acc, tr);
                                        }
                                }
                                pick = __shfl_sync(0xffffffffu, mine_pick, L);
                            } else {
                                const unsigned pos = __ballot_sync(0xffffffffu, gs > 0.0f);
                                if (pos) {
                                    const int L = 31 - __clz(pos);
                                    int lc = -1;
#pragma unroll
                                    for (int jj = 0; jj < 8; ++jj)
                                        if (w[jj] > 0.0f) lc = lo + 8 * g + jj;
                                    lastcol = __shfl_sync(0xffffffffu, lc, L);
                                }
                                acc0 = tf_shfl(endl, 31);
                            }
                        }
                        if (pick < 0) pick = lastcol;
                    }
                    if (pick < 0 && clast >= 0) {
                        // no thread holds t after rounding: this CTA's last positive column
                        float w[8];
                        D.weights(clast, w);
                        int lc = -1;
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj)
                            if (w[jj] > 0.0f) lc = lo + 8 * clast + jj;
                        pick = lc;
                    }
                    if (pick < 0) pick = V - 1;
                    if (lane == 0) P.out_tokens[static_cast<size_t>(b) * R + a] = pick;
                }
            }
            break;
        }
    }
    if (!late && a >= 0) {
        // (4) outputs: drafts 1..a, the emitted token (greedy: written here), -1
        // padding, the count, and the slot_mapping fix-up
        if (lead) {
            int32_t *ot = P.out_tokens + static_cast<size_t>(b) * R;
            for (int i = 0; i < a; ++i) ot[i] = sh.tok[i];
            if (greedy) ot[a] = token;
            for (int i = a + 1; i < R; ++i) ot[i] = -1;
            P.out_count[b] = a;
            if (P.slots) {
                int64_t *sl = P.slots + static_cast<size_t>(b) * R;
                for (int j = a + 1; j < R; ++j) sl[j] = P.pad;
            }
        }
    }
    if (!late && tid == tctl) {
        // rows copied past the rejection and not waited for by the draw (a
        // greedy request, or the stages q did not need) land before exit
        for (int s = 0; s < NS; ++s) {
            int r = -1;
            for (int j = a + 1; j < issued; ++j)
                if (j % NS == s) r = j;
            if (r >= 0 && zmain) wait_copies(&sh.full[s], static_cast<uint32_t>((r / NS) & 1), kWaitLimitNs);
        }
    }
    if (late) {
        // a copy or an exchange outlived its wait: bounded waits for every copy
        // still in flight (the last copy into each stage), so none lands here
        // after exit
        if (tid == tctl) {
            for (int s = 0; s < NS; ++s) {
                int r = -1;
                for (int j = 0; j < issued; ++j)
                    if (j % NS == s) r = j;
                // a stage whose last phase was the plain arrive had its copy land before it
                if (r >= 0 && zmain && s != fake_stage)
                    wait_copies(&sh.full[s], static_cast<uint32_t>((r / NS) & 1), kWaitLimitNs);
            }
            if (drawn_copy) wait_copies(&sh.bar, 0, kWaitLimitNs);
            if (P.status) atomicOr(P.status, SPEC_STATUS_WAIT_TIMEOUT);
        }
    }
    if (bad && P.status) atomicOr(P.status, SPEC_STATUS_NONFINITE);
    if (tid == tctl && P.stats && bytes) atomicAdd(P.stats + 4, bytes);
    cl.sync();   // keep this CTA's shared memory alive until the last remote store into it
}

}  // namespace cc

namespace {
struct CcDevice {
    int ok = 0;
    int sms = 0;
};
CcDevice g_cc_dev[64];

spec_status_t cc_setup(int &sms) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    spec_status_t st = require_sm103(&sms);
    if (st != SPEC_OK) return st;
    if (dev < 0 || dev >= 64) return fail(SPEC_ERR_UNSUPPORTED, "device index out of range%s");
    if (!g_cc_dev[dev].ok) {
        const void *ks[2] = {reinterpret_cast<const void *>(cc::chain_cluster_kernel<2>),
                             reinterpret_cast<const void *>(cc::chain_cluster_kernel<4>)};
        for (int i = 0; i < 2 && e == cudaSuccess; ++i) {
            e = cudaFuncSetAttribute(ks[i], cudaFuncAttributeMaxDynamicSharedMemorySize, cc::kSmemBudget);
            if (e == cudaSuccess) e = cudaFuncSetAttribute(ks[i], cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        }
        if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "chain cluster kernel setup: %s", cudaGetErrorString(e));
        g_cc_dev[dev].ok = 1;
    }
    return SPEC_OK;
}
}  // namespace

// Geometry of the cluster kernel for vocabulary V with C CTAs a request:
// columns per CTA and the ring (stages of one row slice each).  The draw keeps
// row a's logits in its stage and puts q of row a in the others: half of the
// slice in each of two for bf16 logits (so three stages), all of it in one for
// fp32 logits.
struct CcGeom {
    int S, stages;
    size_t stage_bytes, smem;
};

static bool cc_geom(int V, int C, int es, CcGeom &G) {
    G.S = static_cast<int>(((static_cast<long long>(V) + C - 1) / C + 7) / 8 * 8);
    const size_t slice = static_cast<size_t>(G.S) * es;
    const size_t q_part = es == 2 ? static_cast<size_t>((G.S / 8 + 1) / 2) * 32 : static_cast<size_t>(G.S) * 4;
    G.stage_bytes = ((slice > q_part ? slice : q_part) + 127) / 128 * 128;
    const size_t fit = static_cast<size_t>(cc::kSmemBudget) / G.stage_bytes;
    G.stages = static_cast<int>(fit < static_cast<size_t>(cc::kMaxStages) ? fit : static_cast<size_t>(cc::kMaxStages));
    G.smem = G.stages * G.stage_bytes;
    return G.stages >= (es == 2 ? 3 : 2);
}

// Cluster size for a batch of B sampled (or mixed) padded chains with k drafts
// over vocabulary V: the largest C <= 16 whose slices fit in shared memory and
// whose B clusters can all be resident at once; 0 when none qualifies or the
// chains are longer than the kernel takes (the persistent kernel takes the
// batch).
int chain_cluster_size(int B, int k, int V, int es) {
    int sms = 0;
    if (cc_setup(sms) != SPEC_OK || B < 1 || k + 1 > cc::kMaxRowsCC) return 0;
    int dev = 0;
    cudaGetDevice(&dev);
    static std::mutex mu;   // guards the per-device memo of resident-cluster counts below
    for (int C = min(cc::kMaxCluster, sms / B); C >= 1; --C) {
        CcGeom G;
        if (!cc_geom(V, C, es, G)) return 0;   // a smaller cluster has larger slices
        int clusters = 0;
        {
            std::lock_guard<std::mutex> lk(mu);
            static std::vector<std::pair<long long, int>> memo[64];
            const long long key = (static_cast<long long>(es) << 40) | (static_cast<long long>(C) << 32) |
                                  static_cast<long long>(G.smem);
            bool found = false;
            for (auto &kv : memo[dev])
                if (kv.first == key) {
                    clusters = kv.second;
                    found = true;
                }
            if (!found) {
                cudaLaunchConfig_t cfg;
                memset(&cfg, 0, sizeof cfg);
                cfg.gridDim = dim3(static_cast<unsigned>(B) * static_cast<unsigned>(C));
                cfg.blockDim = dim3(cc::kThreads);
                cfg.dynamicSmemBytes = G.smem;
                cudaLaunchAttribute attr[1];
                attr[0].id = cudaLaunchAttributeClusterDimension;
                attr[0].val.clusterDim.x = static_cast<unsigned>(C);
                attr[0].val.clusterDim.y = 1;
                attr[0].val.clusterDim.z = 1;
                cfg.attrs = attr;
                cfg.numAttrs = 1;
                const cudaError_t e =
                    es == 2 ? cudaOccupancyMaxActiveClusters(&clusters, cc::chain_cluster_kernel<2>, &cfg)
                            : cudaOccupancyMaxActiveClusters(&clusters, cc::chain_cluster_kernel<4>, &cfg);
                if (e != cudaSuccess) {
                    cudaGetLastError();
                    clusters = 0;
                }
                memo[dev].push_back({key, clusters});
            }
        }
        if (clusters >= B) return C;
    }
    return 0;
}

spec_status_t launch_chain_cluster(const void *target_logits, spec_dtype_t dtype, const float *draft_probs,
                                   const int32_t *draft_tokens, const float *temperature, const float *u_accept,
                                   const float *u_sample, int B, int k, int V, int32_t *out_tokens,
                                   int32_t *out_num_accepted, int64_t *slot_mapping, int64_t padding_slot_id,
                                   int32_t *d_status, void *workspace, int C, void *stream) {
    int sms = 0;
    spec_status_t st = cc_setup(sms);
    if (st != SPEC_OK) return st;
    const int es = dtype == SPEC_BF16 ? 2 : 4;
    if (C < 1 || C > cc::kMaxCluster) return fail(SPEC_ERR_INVALID_ARG, "cluster size out of range%s");
    cc::Params P;
    memset(&P, 0, sizeof P);
    P.logits = target_logits;
    P.q = draft_probs;
    P.tokens = draft_tokens;
    P.temperature = temperature;
    P.u_accept = u_accept;
    P.u_sample = u_sample;
    P.out_tokens = out_tokens;
    P.out_count = out_num_accepted;
    P.slots = slot_mapping;
    P.pad = padding_slot_id;
    P.status = d_status;
    P.stats = static_cast<unsigned long long *>(workspace);
    P.B = B;
    P.k = k;
    P.V = V;
    P.C = C;
    CcGeom G;
    if (!cc_geom(V, C, es, G) || k + 1 > cc::kMaxRowsCC) return fail(SPEC_ERR_INVALID_ARG, "cluster geometry%s");
    P.S = G.S;
    P.stages = G.stages;
    P.stage_bytes = G.stage_bytes;
    P.smem = G.smem;
    P.zbulk = (static_cast<long long>(V) * es) % 16 == 0;
    P.qbulk = V % 4 == 0;
    P.wait_ns = wait_limit_ns();
    P.logits_end = reinterpret_cast<unsigned long long>(target_logits) +
                   static_cast<unsigned long long>(B) * (k + 1) * static_cast<unsigned long long>(V) * es;
    P.q_end = draft_probs ? reinterpret_cast<unsigned long long>(draft_probs) +
                                static_cast<unsigned long long>(B) * k * static_cast<unsigned long long>(V) * 4
                          : 0ull;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(static_cast<unsigned>(B) * static_cast<unsigned>(C));
    cfg.blockDim = dim3(cc::kThreads);
    cfg.dynamicSmemBytes = G.smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(C);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = es == 2 ? cudaLaunchKernelEx(&cfg, cc::chain_cluster_kernel<2>, P)
                            : cudaLaunchKernelEx(&cfg, cc::chain_cluster_kernel<4>, P);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "chain cluster launch: %s", cudaGetErrorString(e));
    return SPEC_OK;
}

}  // namespace sv
