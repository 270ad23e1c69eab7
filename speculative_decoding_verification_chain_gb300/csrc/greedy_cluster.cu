// greedy_cluster.cu -- greedy verification of padded chains and token trees by
// a persistent grid of thread-block clusters.
//
// What it computes is the greedy step of the persistent verify kernel
// (EAGLE-3 review, the small-draft section: a draft token is accepted iff it
// is the target argmax, lowest index on ties; the first rejection ends a chain
// and emits that row's argmax; all drafts accepted emits the argmax of the
// last row as a bonus token.  For a tree (the EAGLE review's tree attention):
// a node is accepted iff its parent is and its token is the argmax of the
// parent's row; the deepest accepted node, smallest index on ties, is chosen).
//
// Work.  A unit is one row (node n of request b); units are numbered
// node-major (u = n * B + b), so parents are taken before their children.
// Each cluster of C CTAs takes units one at a time from a global counter; CTA
// r of the cluster streams columns [r * S, r * S + S) of the unit's row through
// a ring of three bulk-copy stages, and every streaming warp sends its argmax
// candidate straight to the cluster's first CTA (st.async into its shared
// memory), where an epilogue warp combines the row and publishes it.  Each SM
// streams a quarter (or less) of a row, so a row resolves in about the time one
// SM streams 64 KiB: decisions arrive while their children are still queued.
//
// Roles (416 threads per CTA):
//   * warp 0, copier (every CTA): takes the cluster's work items in order and
//     streams its slice of each row into the ring, unless the row's node has
//     died since the item went out (its dead-mask word, loaded while the stage
//     frees): then its warps send a marker, and the epilogue drops the row;
//   * warp 1, dispatcher (first CTA): claims units, drops those whose node is
//     already known rejected (a per-request mask of dead nodes, loaded while
//     the item's flow-control wait is in flight) and sends the rest to every
//     copier;
//   * warps 2..4, epilogues (first CTA): per row, the argmax over the cluster's
//     candidates, the row's state, the dead mask of the children whose tokens
//     differ from it, and the resolved mask; the row that leaves no node
//     undecided (every node resolved or dead) finalises the request;
//   * warps 5..12, streaming (every CTA): the argmax of each stage.
// Per request one 64-bit word records the resolved rows and the dead nodes
// (two words past 32 rows).  A node is dead when an edge on its root path is
// rejected; once every node not dead is resolved, the nodes not dead are
// exactly the accepted ones.
//
// Every wait is bounded (the caller's limit); a wait that runs out marks the
// CTA aborted, reports SPEC_STATUS_WAIT_TIMEOUT and ends that warp's loop; the
// copier waits (with the default limit) for its copies in flight before exit,
// and no CTA leaves before the cluster barrier.
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

namespace cg = cooperative_groups;

namespace sv {
namespace gc {

constexpr int kMaxC = 16;
constexpr int kStreamWarps = 8;
constexpr int kEpiWarps = 3;
constexpr int kWarpCopy = 0, kWarpDisp = 1, kWarpEpi = 2, kWarpStream = 2 + kEpiWarps;
constexpr int kThreads = 32 * (kWarpStream + kStreamWarps);
constexpr int kStreamThreads = 32 * kStreamWarps;
constexpr int kStages = 3;
constexpr int kItems = 2;      // work items queued per copier
constexpr int kResQ = 8;       // rows whose candidates the first CTA holds
constexpr int kMaxBatch = 2;   // units claimed at once (after rounds of dead units): live ones stay with the cluster
constexpr int kMaxR = 64;      // rows per request (the masks are 64-bit)
constexpr int kSmemBudget = 200 * 1024;
constexpr uint32_t kResolved = 0x80000000u;
constexpr uint32_t kSkipped = 0xfffffffeu;   // the candidate column of a row a CTA found dead
constexpr unsigned long long kWaitLimitNs = 500000000ull;   // copies in flight at exit

struct Params {
    const uint8_t *logits;        // [B, R, V] bf16 bits or fp32
    const int32_t *tokens;        // [B, R-1]: token of node n at column n-1
    int32_t *out_tokens;          // [B, D+1]
    int32_t *out_count;           // [B]: chains a, trees depth + 1
    int32_t *out_path;            // [B, D+1] (trees) or null
    int64_t *slots;               // [B, R] (chains) or null: slot_mapping fix-up
    int64_t pad;
    int32_t *status;
    unsigned long long *stats;    // workspace diagnostic counters
    uint32_t *ctr;                // [0] claims, [1] CTAs finished
    unsigned long long *rmask;    // [B] resolved rows (packed: and dead nodes << 32)
    unsigned long long *dmask;    // [B] dead nodes (R > 32)
    uint32_t *fin;                // [B] finalised
    uint32_t *rowstate;           // [B, R] kResolved | argmax
    uint32_t *reset_base;         // counter region cleared by the last CTA out
    int reset_words;
    unsigned long long wait_ns;
    unsigned long long logits_end;
    unsigned long long stage_bytes;
    int B, R, V, D, C, S, G, tree, zbulk;
    int packed;                       // R <= 32: one word per request, resolved rows low, dead nodes high
    int8_t parent[kMaxR];
    uint8_t depth[kMaxR];
    uint8_t kid_off[kMaxR + 1];
    uint8_t kid_list[kMaxR];
    unsigned long long desc[kMaxR];   // node n and its descendants
};

struct Shared {
    uint64_t full[kStages], empty[kStages];
    uint64_t item_full[kItems], item_empty[kItems];
    uint64_t res_full[kResQ], res_free[kResQ];
    uint64_t rec_full[kResQ];         // first CTA: the slot's item record is written
    int2 items[kItems];               // (b, n); b < 0 ends the work
    int4 stage_item[kStages];         // (b, n, item number, skipped); b < 0 ends the work
    int2 itemrec[kResQ];              // first CTA: (b, n) of the item whose candidates fill the slot
    uint2 res[kResQ][kMaxC * kStreamWarps];   // first CTA: (value bits, column) per streaming warp
    int path[kEpiWarps][kMaxR];       // finalisation scratch per epilogue warp
    int abort;
    int last;
};

// ------------------------------------------------------------ device helpers
__device__ __forceinline__ void remote_arrive(uint64_t *bar, int rank) {
    const uint32_t a = mapa_u32(smem_u32(bar), rank);
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(a) : "memory");
}

__device__ __forceinline__ void st_async_u2(uint32_t dst, uint32_t x, uint32_t y, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];" ::"r"(dst),
                 "r"(x), "r"(y), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned long long atom_or_acqrel_u64(unsigned long long *p, unsigned long long v) {
    unsigned long long old;
    asm volatile("atom.acq_rel.gpu.global.or.b64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
    return old;
}

__device__ __forceinline__ uint32_t atom_add_acqrel(uint32_t *p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void st_relaxed_u32(uint32_t *p, uint32_t v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Bounded wait on a phase of a barrier in this CTA's shared memory (cluster
// scope: remote stores and arrivals complete some of them).
__device__ __forceinline__ bool wait_phase(uint64_t *bar, uint32_t parity, unsigned long long limit) {
    if (limit == 0) return mbar_test_wait_cluster(bar, parity);
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait_cluster(bar, parity))
        if (globaltimer() - t0 > limit) return false;
    return true;
}

// The same for a barrier only this CTA completes (its copies and arrivals).
__device__ __forceinline__ bool wait_local(uint64_t *bar, uint32_t parity, unsigned long long limit) {
    if (limit == 0) return mbar_test_wait(bar, parity);
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer() - t0 > limit) return false;
    return true;
}

__device__ __forceinline__ void set_status(const Params &P, int bits) {
    if (P.status) atomicOr(P.status, bits);
}

// NaN-propagating maximum of two packed bf16 pairs.
__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ float fmax_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Packed running maxima of the two halves of a bf16 pair (NaN-propagating),
// with the first group that raised each half to its current value.
__device__ __forceinline__ void bf16x2_record(uint32_t a, uint32_t &pk, int g, int &glo, int &ghi) {
    asm("{\n\t.reg .pred plo, phi;\n\t"
        "setp.gt.bf16x2 plo|phi, %3, %2;\n\t"
        "selp.s32 %0, %4, %0, plo;\n\t"
        "selp.s32 %1, %4, %1, phi;\n\t}"
        : "+r"(glo), "+r"(ghi)
        : "r"(pk), "r"(a), "r"(g));
    pk = bmax2_nan(pk, a);
}

// Argmax step: (ov, oi) replaces (v, i) when larger, or equal at a lower column.
__device__ __forceinline__ void argmax_take(float &v, int &i, float ov, int oi) {
    if (ov > v || (ov == v && static_cast<unsigned>(oi) < static_cast<unsigned>(i))) {
        v = ov;
        i = oi;
    }
}

__device__ __forceinline__ void warp_argmax(float &v, int &i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        argmax_take(v, i, __shfl_xor_sync(0xffffffffu, v, o), __shfl_xor_sync(0xffffffffu, i, o));
}

// Eight logits of group g as floats; groups at or past gbulk come from global
// memory (zg: the slice's first column; -inf past column n).
template <int ES>
__device__ __forceinline__ void group8(const uint8_t *zs, const uint8_t *zg, int g, int gbulk, int n, float x[8],
                                       float &gm) {
    if (g < gbulk) {
        if constexpr (ES == 2) {
            const uint4 w = reinterpret_cast<const uint4 *>(zs)[g];
            const uint32_t m2 = bmax2_nan(bmax2_nan(w.x, w.y), bmax2_nan(w.z, w.w));
            gm = fmax_nan(bf_lo(m2), bf_hi(m2));
            x[0] = bf_lo(w.x); x[1] = bf_hi(w.x); x[2] = bf_lo(w.y); x[3] = bf_hi(w.y);
            x[4] = bf_lo(w.z); x[5] = bf_hi(w.z); x[6] = bf_lo(w.w); x[7] = bf_hi(w.w);
            return;
        } else {
            const float4 a = reinterpret_cast<const float4 *>(zs)[2 * g], c = reinterpret_cast<const float4 *>(zs)[2 * g + 1];
            x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = c.x; x[5] = c.y; x[6] = c.z; x[7] = c.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int c = 8 * g + j;
            if (c >= n)
                x[j] = -INFINITY;
            else if constexpr (ES == 2)
                x[j] = __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const uint16_t *>(zg) + c)) << 16);
            else
                x[j] = __ldg(reinterpret_cast<const float *>(zg) + c);
        }
    }
    gm = fmax_nan(fmax_nan(fmax_nan(x[0], x[1]), fmax_nan(x[2], x[3])), fmax_nan(fmax_nan(x[4], x[5]), fmax_nan(x[6], x[7])));
}

template <int ES>
__global__ void __launch_bounds__(kThreads, 1) greedy_cluster_kernel(const __grid_constant__ Params P) {
    extern __shared__ __align__(128) uint8_t dyn[];
    __shared__ Shared sh;
    cg::cluster_group cl = cg::this_cluster();
    const int C = P.C;
    const int rank = static_cast<int>(cl.block_rank());
    const int cid = static_cast<int>(blockIdx.x) / C;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool leader = rank == 0;
    const int B = P.B, R = P.R, V = P.V, S = P.S;
    const int lo = rank * S;
    const int n = max(0, min(S, V - lo));          // columns of this CTA
    const int ng = (n + 7) >> 3;
    const uint32_t zmain = P.zbulk ? static_cast<uint32_t>((n * ES) & ~15) : 0u;
    const int gbulk = static_cast<int>(zmain / (8 * ES));
    const int total = B * R;
    const unsigned long long valid = R >= 64 ? ~0ull : ((1ull << R) - 1ull);

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&sh.full[i], 1);
            mbar_init(&sh.empty[i], kStreamWarps);
        }
        for (int i = 0; i < kItems; ++i) {
            mbar_init(&sh.item_full[i], 1);
            mbar_init(&sh.item_empty[i], C);
        }
        for (int i = 0; i < kResQ; ++i) {
            mbar_init(&sh.res_full[i], 1);
            mbar_init(&sh.res_free[i], 1);
            mbar_init(&sh.rec_full[i], 1);
        }
        sh.abort = 0;
        sh.last = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // Every cluster of the grid is resident from the start, so the next kernel
    // may begin launching at once; nothing below touches global memory before
    // the previous kernel in the stream has completed.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __syncthreads();
    cl.sync();   // every CTA's barriers exist before any remote store or arrival
    auto abort_here = [&]() {
        if (lane == 0) {
            sh.abort = 1;
            set_status(P, SPEC_STATUS_WAIT_TIMEOUT);
        }
    };

    bool bad = false;
    if (warp == kWarpCopy) {
        // ------------------------------------------------------------ copier
        int it = 0;                 // ring uses
        int last_use[kStages] = {-1, -1, -1};
        unsigned long long bytes = 0;
        if (lane == 0) {
            for (int j = 0;; ++j) {
                const int s = j % kItems;
                mbar_expect_tx(&sh.item_full[s], 8u);
                if (!wait_phase(&sh.item_full[s], static_cast<uint32_t>((j / kItems) & 1), P.wait_ns)) {
                    abort_here();
                    break;
                }
                const int2 itm = sh.items[s];
                remote_arrive(&sh.item_empty[s], 0);   // the slot may be refilled
                // the node may have died since the item went out: its dead-mask
                // word loads while the stage frees, and a dead row is not copied
                unsigned long long dm = 0;
                if (itm.x >= 0 && itm.y > 0)
                    dm = P.packed ? (ld_relaxed_u64(P.rmask + itm.x) >> 32) : ld_relaxed_u64(P.dmask + itm.x);
                const int st = it % kStages;
                if (it >= kStages &&
                    !wait_local(&sh.empty[st], static_cast<uint32_t>(((it / kStages) - 1) & 1), P.wait_ns)) {
                    abort_here();
                    break;
                }
                if (itm.x < 0) {
                    sh.stage_item[st] = make_int4(-1, 0, 0, 0);
                    mbar_arrive(&sh.full[st]);
                    last_use[st] = -1;   // no copy
                    ++it;
                    break;
                }
                const bool dead = itm.y > 0 && ((dm >> itm.y) & 1ull);
                sh.stage_item[st] = make_int4(itm.x, itm.y, j, dead ? 1 : 0);
                if (zmain && !dead) {
                    fence_proxy_async();
                    mbar_expect_tx(&sh.full[st], zmain);
                    bulk_g2s(dyn + static_cast<size_t>(st) * P.stage_bytes,
                             P.logits + ((static_cast<size_t>(itm.x) * R + itm.y) * V + lo) * ES, zmain, &sh.full[st]);
                    bytes += zmain;
                    last_use[st] = it;
                } else {
                    mbar_arrive(&sh.full[st]);
                    last_use[st] = -1;
                }
                ++it;
            }
            if (sh.abort) {
                // copies still in flight land before this CTA's memory goes away
                for (int s = 0; s < kStages; ++s)
                    if (last_use[s] >= 0)
                        wait_local(&sh.full[s], static_cast<uint32_t>((last_use[s] / kStages) & 1), kWaitLimitNs);
            }
            if (P.stats && bytes) atomicAdd(P.stats + 4, bytes);
        }
        __syncwarp();
    } else if (warp == kWarpDisp) {
        // -------------------------------------------------------- dispatcher
        if (leader) {
            int j = 0;   // items sent
            // Flow control: item j may go out once its queue slot (every copier
            // took item j - kItems) and its candidate slot (the epilogue took
            // item j - kResQ) are free.  Waiting again for the same j returns at once.
            auto flow = [&](bool items) -> bool {
                bool ok = true;
                if (lane == 0) {
                    const int s = j % kItems, rs = j % kResQ;
                    if (items && j >= kItems)
                        ok = wait_phase(&sh.item_empty[s], static_cast<uint32_t>(((j / kItems) - 1) & 1), P.wait_ns);
                    if (ok && j >= kResQ)
                        ok = wait_local(&sh.res_free[rs], static_cast<uint32_t>(((j / kResQ) - 1) & 1), P.wait_ns);
                }
                return __shfl_sync(0xffffffffu, ok, 0) != 0;
            };
            // Item j = (b, n) to every copier (b < 0: the end), after flow(true).
            auto put = [&](int b, int nn) {
                if (lane == 0) {
                    const int s = j % kItems, rs = j % kResQ;
                    sh.itemrec[rs] = make_int2(b, nn);
                    mbar_arrive(&sh.rec_full[rs]);
                    if (b >= 0) mbar_expect_tx(&sh.res_full[rs], 8u * static_cast<uint32_t>(C * kStreamWarps));
                    else mbar_arrive(&sh.res_full[rs]);
                    for (int q = 0; q < C; ++q)
                        st_async_u2(mapa_u32(smem_u32(&sh.items[s]), q), static_cast<uint32_t>(b), static_cast<uint32_t>(nn),
                                    mapa_u32(smem_u32(&sh.item_full[s]), q));
                }
                ++j;
            };
            bool aborted = false;
            // A round: the batch of units claimed during the previous round (lane
            // i < m holds one) has its dead-mask words loaded while the next
            // batch's claim (one atomic) and the flow-control wait are in flight;
            // then its live units go out in unit order.  A batch is one unit, or
            // twice the one before (up to kMaxBatch) after a round with none
            // alive: a cluster keeps every live unit it claims.  The
            // cluster's first unit is its own (claimed statically).
            int u = lane == 0 ? cid : INT_MAX;
            int mn = 1;
            while (!aborted) {
                const bool ok = u < total;
                if (!__any_sync(0xffffffffu, ok)) break;
                const int b = ok ? u % B : 0, nn = ok ? u / B : 0;
                unsigned long long dm = 0;
                if (ok && nn > 0) dm = P.packed ? (ld_acquire_u64(P.rmask + b) >> 32) : ld_acquire_u64(P.dmask + b);
                unsigned base = 0;
                if (lane == 0) base = atomicAdd(P.ctr, static_cast<unsigned>(mn));
                if (!flow(true)) {
                    aborted = true;
                    break;
                }
                unsigned alive = __ballot_sync(0xffffffffu, ok && !((dm >> nn) & 1ull));
                const int mafter = alive ? 1 : min(kMaxBatch, 2 * mn);
                bool first = true;
                while (alive && !aborted) {
                    if (!first && !flow(true)) {
                        aborted = true;
                        break;
                    }
                    first = false;
                    int key = ((alive >> lane) & 1u) ? u : INT_MAX;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) key = min(key, __shfl_xor_sync(0xffffffffu, key, o));
                    const int src = __ffs(__ballot_sync(0xffffffffu, u == key && ((alive >> lane) & 1u))) - 1;
                    alive &= ~(1u << src);
                    put(__shfl_sync(0xffffffffu, b, src), __shfl_sync(0xffffffffu, nn, src));
                }
                base = __shfl_sync(0xffffffffu, base, 0);
                u = lane < mn ? P.G + static_cast<int>(base) + lane : INT_MAX;
                mn = mafter;
            }
            // the end: one item for the copiers, then one marker per other epilogue warp
            if (!aborted) {
                if (flow(true)) put(-1, 0);
                else aborted = true;
            }
            for (int e = 1; e < kEpiWarps && !aborted; ++e) {
                if (!flow(false)) {
                    aborted = true;
                    break;
                }
                if (lane == 0) {
                    const int rs = j % kResQ;
                    sh.itemrec[rs] = make_int2(-1, 0);
                    mbar_arrive(&sh.rec_full[rs]);
                    mbar_arrive(&sh.res_full[rs]);
                }
                ++j;
            }
            if (aborted) abort_here();
        }
    } else if (warp < kWarpStream) {
        // ---------------------------------------------------------- epilogue
        if (leader) {
            const int e = warp - kWarpEpi;
            int *path = sh.path[e];
            for (int j = e;; j += kEpiWarps) {
                const int rs = j % kResQ;
                const uint32_t ph = static_cast<uint32_t>((j / kResQ) & 1);
                // the item's record first: its children's tokens load while the
                // row's candidates are still on their way
                if (!wait_local(&sh.rec_full[rs], ph, P.wait_ns)) {
                    abort_here();
                    break;
                }
                const int2 rec = sh.itemrec[rs];
                const int b = rec.x, nd = rec.y;
                const int k0 = b < 0 ? 0 : (P.tree ? P.kid_off[nd] : nd + 1);
                const int k1 = b < 0 ? 0 : (P.tree ? P.kid_off[nd + 1] : min(nd + 2, R));
                int kt[2] = {-1, -1}, kc[2] = {0, 0};   // lanes hold children q and q + 32
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int q = k0 + lane + 32 * h;
                    if (q < k1) {
                        kc[h] = P.tree ? P.kid_list[q] : q;
                        kt[h] = __ldg(P.tokens + static_cast<size_t>(b) * (R - 1) + kc[h] - 1);
                    }
                }
                if (!wait_phase(&sh.res_full[rs], ph, P.wait_ns)) {
                    abort_here();
                    break;
                }
                float v = -INFINITY;
                int g = INT_MAX;
                bool skipped = false;
                if (b >= 0)
                    for (int q = lane; q < C * kStreamWarps; q += 32) {
                        const uint2 c = sh.res[rs][q];
                        skipped |= c.y == kSkipped;
                        argmax_take(v, g, __uint_as_float(c.x), static_cast<int>(c.y));
                    }
                skipped = __any_sync(0xffffffffu, skipped);
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.res_free[rs]);
                if (b < 0) break;
                if (skipped) continue;   // its node is dead: nothing waits for the row
                warp_argmax(v, g);
                if (!(v > -INFINITY) && lane == 0) set_status(P, SPEC_STATUS_NONFINITE);   // a row -inf throughout
                const int arg = (g >= 0 && g < V) ? g : 0;
                // children whose tokens differ from the argmax: their subtrees are dead
                unsigned long long dead = 0;
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    if (k0 + lane + 32 * h < k1 && kt[h] != arg) dead |= P.desc[kc[h]];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) dead |= __shfl_xor_sync(0xffffffffu, dead, o);
                unsigned long long dm = 0, now = 0;
                if (lane == 0) {
                    st_relaxed_u32(P.rowstate + static_cast<size_t>(b) * R + nd, kResolved | static_cast<uint32_t>(arg));
                    if (P.packed) {
                        // one word: resolved rows and dead nodes change together
                        const unsigned long long w = atom_or_acqrel_u64(P.rmask + b, (dead << 32) | (1ull << nd)) |
                                                     (dead << 32) | (1ull << nd);
                        now = w & 0xffffffffull;
                        dm = w >> 32;
                    } else {
                        if (dead) atomicOr(P.dmask + b, dead);
                        // acq_rel: the dead bits and the row state above are ordered before it
                        now = atom_or_acqrel_u64(P.rmask + b, 1ull << nd) | (1ull << nd);
                        dm = ld_acquire_u64(P.dmask + b);
                    }
                }
                dm = __shfl_sync(0xffffffffu, dm, 0);
                now = __shfl_sync(0xffffffffu, now, 0);
                bool first = false;
                if ((~dm & ~now & valid) == 0ull && lane == 0) first = atomicExch(P.fin + b, 1u) == 0u;
                if (!__shfl_sync(0xffffffffu, first, 0)) continue;
                __syncwarp();   // the whole warp reads after lane 0's acquire
                // -------- finalise request b: the accepted nodes are those not dead
                const unsigned long long acc = ~dm & valid;
                int key = -1;   // depth * 256 + (255 - node): deepest, then smallest index
                for (int c = lane; c < R; c += 32)
                    if ((acc >> c) & 1ull) key = max(key, static_cast<int>(P.depth[c]) * 256 + (255 - c));
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) key = max(key, __shfl_xor_sync(0xffffffffu, key, o));
                const int best = 255 - (key & 255), d = key >> 8;
                if (lane == 0) {
                    int x = best;
                    for (int i = d; i >= 0; --i) {
                        path[i] = x;
                        x = P.parent[x];
                    }
                }
                __syncwarp();
                const uint32_t rsb = P.rowstate[static_cast<size_t>(b) * R + best];
                const int emit = (rsb & kResolved) ? static_cast<int>(rsb & 0x7fffffffu) : 0;
                int32_t *ot = P.out_tokens + static_cast<size_t>(b) * (P.D + 1);
                for (int i = lane; i <= P.D; i += 32) {
                    int t = -1;
                    if (i < d) t = __ldg(P.tokens + static_cast<size_t>(b) * (R - 1) + path[i + 1] - 1);
                    else if (i == d) t = emit;
                    ot[i] = t;
                    if (P.out_path) P.out_path[static_cast<size_t>(b) * (P.D + 1) + i] = i <= d ? path[i] : -1;
                }
                if (P.slots)
                    for (int i = d + 1 + lane; i < R; i += 32) P.slots[static_cast<size_t>(b) * R + i] = P.pad;
                // a token outside [0, V) anywhere in the request is reported
                bool range = false;
                for (int i = lane; i < R - 1; i += 32) {
                    const int t = __ldg(P.tokens + static_cast<size_t>(b) * (R - 1) + i);
                    range |= t < 0 || t >= V;
                }
                if (__any_sync(0xffffffffu, range) && lane == 0) set_status(P, SPEC_STATUS_TOKEN_RANGE);
                if (lane == 0) P.out_count[b] = P.tree ? d + 1 : d;
            }
        }
    } else {
        // --------------------------------------------------------- streaming
        const int w = warp - kWarpStream;
        const int sid = tid - 32 * kWarpStream;
        for (int it = 0;; ++it) {
            const int st = it % kStages;
            if (!wait_local(&sh.full[st], static_cast<uint32_t>((it / kStages) & 1), P.wait_ns)) {
                abort_here();
                break;
            }
            const int4 si = sh.stage_item[st];
            if (si.x < 0) break;
            if (si.w) {
                // a row found dead at its copy: a marker instead of a candidate
                if (lane == 0) {
                    const int rs = si.z % kResQ;
                    st_async_u2(mapa_u32(smem_u32(&sh.res[rs][rank * kStreamWarps + w]), 0), __float_as_uint(-INFINITY),
                                kSkipped, mapa_u32(smem_u32(&sh.res_full[rs]), 0));
                    mbar_arrive(&sh.empty[st]);
                }
                continue;
            }
            const uint8_t *zs = dyn + static_cast<size_t>(st) * P.stage_bytes;
            const uint8_t *zg = P.logits + ((static_cast<size_t>(si.x) * R + si.y) * V + lo) * ES;
            float best = -INFINITY;
            int bi = INT_MAX;
            bool nan = false;
            if constexpr (ES == 2) {
                // branch-free packed maxima over the groups in shared memory, four
                // loads in flight per thread; the exact column is found in the
                // stage before it is released
                constexpr int K = 4;
                uint32_t pk = 0xff80ff80u;
                int glo = -1, ghi = -1;
                const uint4 *z4 = reinterpret_cast<const uint4 *>(zs);
                for (int g0 = sid; g0 < gbulk; g0 += K * kStreamThreads) {
                    uint4 r[K];
#pragma unroll
                    for (int q = 0; q < K; ++q)
                        if (g0 + q * kStreamThreads < gbulk) r[q] = z4[g0 + q * kStreamThreads];
#pragma unroll
                    for (int q = 0; q < K; ++q)
                        if (g0 + q * kStreamThreads < gbulk)
                            bf16x2_record(bmax2_nan(bmax2_nan(r[q].x, r[q].y), bmax2_nan(r[q].z, r[q].w)), pk,
                                          g0 + q * kStreamThreads, glo, ghi);
                }
                const float vlo = bf_lo(pk), vhi = bf_hi(pk);
                nan |= !(vlo == vlo) || !(vhi == vhi) || vlo == INFINITY || vhi == INFINITY;
                const float v = fmaxf(vlo, vhi);
                if (v > -INFINITY) {
                    // the first column holding v: a lo position of group glo or a hi position of group ghi
                    int col = INT_MAX;
                    if (glo >= 0 && vlo == v) {
                        const uint4 w = z4[glo];
                        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
                        int j = 8;
#pragma unroll
                        for (int q = 3; q >= 0; --q)
                            if (bf_lo(ww[q]) == v) j = 2 * q;
                        col = lo + 8 * glo + j;
                    }
                    if (ghi >= 0 && vhi == v) {
                        const uint4 w = z4[ghi];
                        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
                        int j = 8;
#pragma unroll
                        for (int q = 3; q >= 0; --q)
                            if (bf_hi(ww[q]) == v) j = 2 * q + 1;
                        col = min(col, lo + 8 * ghi + j);
                    }
                    best = v;
                    bi = col;
                }
                // groups the bulk copy does not cover (a row end off the 16-byte grid)
                for (int g = gbulk + sid; g < ng; g += kStreamThreads) {
                    float x[8], gm;
                    group8<ES>(zs, zg, g, gbulk, n, x, gm);
                    nan |= !(gm == gm) || gm == INFINITY;
                    if (gm > best) {
                        int j = 7;
#pragma unroll
                        for (int q = 7; q >= 0; --q)
                            if (x[q] == gm) j = q;
                        best = gm;
                        bi = lo + 8 * g + j;
                    }
                }
            } else {
                for (int g = sid; g < ng; g += kStreamThreads) {
                    float x[8], gm;
                    group8<ES>(zs, zg, g, gbulk, n, x, gm);
                    nan |= !(gm == gm) || gm == INFINITY;
                    if (gm > best) {
                        int j = 7;
#pragma unroll
                        for (int q = 7; q >= 0; --q)
                            if (x[q] == gm) j = q;
                        best = gm;
                        bi = lo + 8 * g + j;
                    }
                }
            }
            bad |= nan;
            warp_argmax(best, bi);
            __syncwarp();
            if (lane == 0) {
                const int rs = si.z % kResQ;
                st_async_u2(mapa_u32(smem_u32(&sh.res[rs][rank * kStreamWarps + w]), 0), __float_as_uint(best),
                            static_cast<uint32_t>(bi), mapa_u32(smem_u32(&sh.res_full[rs]), 0));
                mbar_arrive(&sh.empty[st]);
            }
        }
    }
    if (bad) set_status(P, SPEC_STATUS_NONFINITE);
    __syncthreads();
    cl.sync();   // no CTA leaves while a remote store or arrival may still target it
    if (tid == 0) sh.last = atom_add_acqrel(P.ctr + 1, 1u) == gridDim.x - 1;
    __syncthreads();
    if (sh.last) {
        // every other CTA is done with the counters: clear them for the next call
        for (int i = tid; i < P.reset_words; i += kThreads) P.reset_base[i] = 0u;
    }
}

}  // namespace gc

namespace {
struct GcDevice {
    int ok = 0;
};
GcDevice g_gc_dev[64];

spec_status_t gc_setup(int &sms) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    spec_status_t st = require_sm103(&sms);
    if (st != SPEC_OK) return st;
    if (dev < 0 || dev >= 64) return fail(SPEC_ERR_UNSUPPORTED, "device index out of range%s");
    if (!g_gc_dev[dev].ok) {
        const void *ks[2] = {reinterpret_cast<const void *>(gc::greedy_cluster_kernel<2>),
                             reinterpret_cast<const void *>(gc::greedy_cluster_kernel<4>)};
        for (int i = 0; i < 2 && e == cudaSuccess; ++i) {
            e = cudaFuncSetAttribute(ks[i], cudaFuncAttributeMaxDynamicSharedMemorySize, gc::kSmemBudget);
            if (e == cudaSuccess) e = cudaFuncSetAttribute(ks[i], cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        }
        if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "greedy cluster kernel setup: %s", cudaGetErrorString(e));
        g_gc_dev[dev].ok = 1;
    }
    return SPEC_OK;
}

// Columns per CTA and the stage size for cluster size C: three stages of one
// row slice each must fit the shared-memory budget.
bool gc_geom(int V, int C, int es, int &S, size_t &stage_bytes) {
    S = static_cast<int>(((static_cast<long long>(V) + C - 1) / C + 7) / 8 * 8);
    stage_bytes = (static_cast<size_t>(S) * es + 127) / 128 * 128;
    return stage_bytes * gc::kStages <= static_cast<size_t>(gc::kSmemBudget);
}

// Clusters of C CTAs resident at once (memoised per device).
int gc_resident(int C, int es, size_t smem) {
    int dev = 0;
    cudaGetDevice(&dev);
    static std::mutex mu;
    static std::vector<std::pair<long long, int>> memo[64];
    std::lock_guard<std::mutex> lk(mu);
    const long long key = (static_cast<long long>(es) << 40) | (static_cast<long long>(C) << 32) | static_cast<long long>(smem);
    for (auto &kv : memo[dev])
        if (kv.first == key) return kv.second;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(static_cast<unsigned>(C));
    cfg.blockDim = dim3(gc::kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(C);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    const cudaError_t e = es == 2 ? cudaOccupancyMaxActiveClusters(&clusters, gc::greedy_cluster_kernel<2>, &cfg)
                                  : cudaOccupancyMaxActiveClusters(&clusters, gc::greedy_cluster_kernel<4>, &cfg);
    if (e != cudaSuccess) {
        cudaGetLastError();
        clusters = 0;
    }
    memo[dev].push_back({key, clusters});
    return clusters;
}
}  // namespace

// See common.h.
spec_status_t launch_greedy_cluster(const GreedyClusterArgs &A, void *stream, bool &launched) {
    launched = false;
    // Greedy trees always; greedy padded chains with fewer than two rows per SM
    // (where the persistent kernel would split rows), or every one on path 2.
    // With two rows per SM or more the persistent kernel's whole-row units
    // stream faster (B = 64, k = 5, V = 128256: 20.5 against 22.4 us; at B = 48
    // the grid takes 19.9 against 21.7, at B = 8 10.4 against 12.1).
    const int path = tuning_path();
    if (path == 1 || A.R < 2 || A.R > gc::kMaxR) return SPEC_OK;
    int sms = 0;
    spec_status_t st = gc_setup(sms);
    if (st != SPEC_OK) return st;
    if (!A.parent && path != 2 && static_cast<long long>(A.B) * A.R >= 2ll * sms) return SPEC_OK;
    const int es = A.dtype == SPEC_BF16 ? 2 : 4;
    int C = 0, S = 0;
    size_t stage_bytes = 0;
    for (int c : {4, 8, 16})
        if (gc_geom(A.V, c, es, S, stage_bytes)) {
            C = c;
            break;
        }
    if (C == 0) return SPEC_OK;
    const size_t smem = stage_bytes * gc::kStages;
    int G = sms / C;
    const int res = gc_resident(C, es, smem);
    if (res < G) G = res;
    if (G < 1) return SPEC_OK;
    gc::Params P;
    memset(&P, 0, sizeof P);
    P.logits = static_cast<const uint8_t *>(A.logits);
    P.tokens = A.tokens;
    P.out_tokens = A.out_tokens;
    P.out_count = A.out_count;
    P.out_path = A.out_path;
    P.slots = A.slots;
    P.pad = A.pad;
    P.status = A.status;
    P.stats = A.stats;
    P.ctr = A.ctr;
    P.rmask = A.rmask;
    P.dmask = A.dmask;
    P.fin = A.fin;
    P.rowstate = A.rowstate;
    P.reset_base = A.reset_base;
    P.reset_words = A.reset_words;
    P.wait_ns = wait_limit_ns();
    P.B = A.B;
    P.R = A.R;
    P.V = A.V;
    P.D = A.D;
    P.C = C;
    P.S = S;
    P.G = G;
    P.tree = A.parent ? 1 : 0;
    P.packed = A.R <= 32;
    P.zbulk = (static_cast<long long>(A.V) * es) % 16 == 0;
    P.stage_bytes = stage_bytes;
    P.logits_end = reinterpret_cast<unsigned long long>(A.logits) +
                   static_cast<unsigned long long>(A.B) * A.R * static_cast<unsigned long long>(A.V) * es;
    // the tree (a chain is the tree whose node n has parent n-1)
    int cnt[gc::kMaxR + 1] = {0};
    for (int nd = 0; nd < A.R; ++nd) {
        const int p = nd == 0 ? -1 : (A.parent ? A.parent[nd] : nd - 1);
        P.parent[nd] = static_cast<int8_t>(p);
        P.depth[nd] = static_cast<uint8_t>(nd == 0 ? 0 : P.depth[p] + 1);
        if (p >= 0) ++cnt[p];
    }
    int off = 0;
    for (int nd = 0; nd < A.R; ++nd) {
        P.kid_off[nd] = static_cast<uint8_t>(off);
        off += cnt[nd];
        cnt[nd] = P.kid_off[nd];
    }
    P.kid_off[A.R] = static_cast<uint8_t>(off);
    for (int nd = 1; nd < A.R; ++nd) P.kid_list[cnt[P.parent[nd]]++] = static_cast<uint8_t>(nd);
    for (int nd = A.R - 1; nd >= 0; --nd) {
        P.desc[nd] |= 1ull << nd;
        if (nd > 0) P.desc[P.parent[nd]] |= P.desc[nd];
    }
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(static_cast<unsigned>(G * C));
    cfg.blockDim = dim3(gc::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(C);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = es == 2 ? cudaLaunchKernelEx(&cfg, gc::greedy_cluster_kernel<2>, P)
                            : cudaLaunchKernelEx(&cfg, gc::greedy_cluster_kernel<4>, P);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "greedy cluster launch: %s", cudaGetErrorString(e));
    launched = true;
    return SPEC_OK;
}

}  // namespace sv
