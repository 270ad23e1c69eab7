// spec_verify.cu -- GB300 (sm_103a) verify-and-accept for speculative decoding.
//
// One persistent kernel verifies chains (greedy or sampled, per request) and
// greedy token trees.  A chain is handled as a tree whose node n has parent
// n-1, so both share one scheduler:
//
//   * Work is cut into units.  An "A unit" is one chunk of one logits row of
//     one request; a "B unit" is one chunk of the rejected row of a sampled
//     request (residual pass).  Units are numbered row-major over
//     (node, request, chunk) so that every row's chunks are claimed together
//     and a parent row is claimed long before its children.
//   * Each block claims units with one global atomic, checks whether the row
//     is still needed (a row is needed only if its node can still be
//     accepted: every ancestor edge either unresolved or matching), streams
//     the chunk into shared memory with one bulk-async copy (cp.async.bulk
//     completing on an mbarrier) and reduces it: argmax (greedy) or max and
//     sum of exp2 (sampled) plus 256-element block sums for the inverse CDF.
//   * The last unit of a row (arrival counter) combines the chunk partials
//     and resolves the row: its argmax, or its softmax statistics and the
//     accept test min(1, p/q) of the one child.  The last unit of a request
//     walks the tree, picks the deepest accepted node and writes the outputs;
//     a sampled request rejected at row a then releases its B units, whose
//     last one locates u * (residual mass) in the block sums and scans one
//     256-element block for the token.  No row of the residual max(0, p - q)
//     is ever written to memory.
//   * Rows of a node that is already known to be rejected are skipped without
//     being read, so the logits actually streamed approach the bytes the
//     method needs (rows up to the first rejection).
//
// Every inter-block wait is bounded by a wall-clock limit and reports
// SPEC_STATUS_WAIT_TIMEOUT instead of hanging.  The last block to exit clears
// the workspace counters, so the next call (or graph replay) starts clean.
//
// Arithmetic: logits are widened to fp32 exactly; exponentials use the
// hardware ex2 approximation on (z - max) * log2(e)/T; chunk combinations
// and the inverse-CDF prefix across blocks are in fp64.

#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "spec_verify.h"

namespace sv {

// ---------------------------------------------------------------- config --
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kBlk = 256;                 // canonical block: 32 lanes x 8 elements
constexpr int kChunkA = 8192;             // elements per A unit (row chunk)
constexpr int kChunkB = 4096;             // elements per B unit (residual chunk)
constexpr int kQOff = 16384 + 64;         // q area offset inside a stage (B units)
constexpr int kStageBytes = 32768 + 128;  // z chunk (<= 32 KiB) or z + q of a B unit
constexpr int kMaxRows = SPEC_MAX_ROWS;
constexpr uint32_t kResolved = 0x80000000u;
constexpr uint32_t kIdxMask = 0x3fffffffu;
constexpr uint32_t kDecided = 0x80000000u;
constexpr uint32_t kNeedsResidual = 0x40000000u;
constexpr unsigned long long kWaitLimitNs = 500000000ull;   // 0.5 s

enum UnitKind : int { kEnd = 0, kALoad = 1, kASkip = 2, kBLoad = 3, kBSkip = 4, kBWait = 5 };

struct RowStat {
    float m;      // row max of raw logits
    float pad;
    double S;     // sum_j exp2((z_j - m) * c2)
};

struct Partial {
    float v;      // chunk max
    int32_t idx;  // argmax (row index), greedy only
    double s;     // sum of exp2((z - v) * c2) over the chunk, sampled only
};

struct Params {
    const uint8_t *logits;
    const float *q;
    const int32_t *tokens;       // [B, R-1]
    const float *temperature;    // [B] or null
    const float *u_accept;       // [B, R-1] or null
    const float *u_sample;       // [B, R] or null
    int32_t *out_tokens;         // [B, D+1]
    int32_t *out_count;          // chain: num_accepted, tree: length
    int32_t *out_path;           // tree only
    int32_t *status;             // may be null
    // workspace
    unsigned long long *stats;   // [8], never cleared by the kernel
    uint32_t *ctrl;              // [32]: 0 claim counter, 1 exit counter
    uint32_t *row_done;          // [B*R]
    uint32_t *rowstate;          // [B*R]
    uint32_t *req_done;          // [B]
    uint32_t *req_state;         // [B]
    uint32_t *res_done;          // [B]
    uint32_t *reset_base;
    uint32_t reset_words;
    RowStat *rowstat;            // [B*R]
    Partial *partial;            // [B*R*nca]
    float *bsumA;                // [B*R*nblk]
    float *bsumB;                // [B*nblk]
    unsigned long long logits_end;  // one past the last logits byte (address)
    unsigned long long q_end;
    int B, R, V, D;
    int esize;
    int nca, ncb, nblk;
    int units_a, units_total;
    int tree;
    int16_t parent[kMaxRows];
    uint8_t depth[kMaxRows];
};

struct Unit {
    int kind;
    int b, n, c;
    int cnt;            // elements in this chunk
    int sh, tail;       // z: byte shift of element 0 in the stage, elements [tail,cnt) from global
    int shq, tailq;     // q (B units)
    uint32_t bytes;     // bulk bytes expected on the stage barrier
    float c2;           // log2(e) / T, or 0 for greedy
    float m;            // row max (B units)
    float invS;         // 1 / S (B units)
    const uint8_t *gz;  // global address of element 0 of the z chunk
    const uint8_t *gq;  // global address of element 0 of the q chunk
};

// ------------------------------------------------------- ptx wrappers --
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t phase) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(phase)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src_gmem, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t atom_add_acqrel(uint32_t *p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// 2^x by the SFU approximation (flushes results below 2^-126 to zero).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void set_status(const Params &P, int bits) {
    if (P.status) atomicOr(P.status, bits);
}

// ------------------------------------------------------------ weights --
// The two per-element weights of the inverse CDF.  Written with explicit
// rounding intrinsics so every call site evaluates them bit-identically.
__device__ __forceinline__ float w_exp(float z, float M, float c2) {
    return ex2(__fmul_rn(__fsub_rn(z, M), c2));
}

__device__ __forceinline__ float w_res(float z, float qv, float m, float c2, float invS) {
    float p = __fmul_rn(ex2(__fmul_rn(__fsub_rn(z, m), c2)), invS);
    return fmaxf(__fsub_rn(p, qv), 0.0f);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t nonfinite_bf16x2(uint32_t w) {
    return __vcmpeq2(w & 0x7f807f80u, 0x7f807f80u);
}

__device__ __forceinline__ uint32_t nonfinite_f32(uint32_t w) {
    return (w & 0x7f800000u) == 0x7f800000u;
}

// Element view of one chunk: elements [0, tail) live in shared memory at s,
// elements [tail, cnt) are read from global memory at g.
struct View {
    const uint8_t *s;
    const uint8_t *g;
    int cnt, tail;
    bool aligned;
};

template <int ES>
__device__ __forceinline__ float ld_one(const View &v, int e, uint32_t &bad) {
    if (ES == 2) {
        uint16_t h = (e < v.tail) ? *reinterpret_cast<const uint16_t *>(v.s + 2 * e)
                                  : __ldg(reinterpret_cast<const unsigned short *>(v.g + 2 * e));
        bad |= ((h & 0x7f80u) == 0x7f80u);
        return __uint_as_float(static_cast<uint32_t>(h) << 16);
    } else {
        uint32_t w = (e < v.tail) ? *reinterpret_cast<const uint32_t *>(v.s + 4 * e)
                                  : __ldg(reinterpret_cast<const unsigned int *>(v.g + 4 * e));
        bad |= nonfinite_f32(w);
        return __uint_as_float(w);
    }
}

// Loads the 8 elements [e0, e0+8) of a view; returns how many are valid.
template <int ES>
__device__ __forceinline__ int load8(const View &v, int e0, float x[8], uint32_t &bad) {
    int nv = v.cnt - e0;
    if (nv <= 0) return 0;
    if (v.aligned && e0 + 8 <= v.tail) {
        if (ES == 2) {
            uint4 w = *reinterpret_cast<const uint4 *>(v.s + 2 * e0);
            bad |= nonfinite_bf16x2(w.x) | nonfinite_bf16x2(w.y) | nonfinite_bf16x2(w.z) | nonfinite_bf16x2(w.w);
            x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x);
            x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
            x[4] = bf16_lo(w.z); x[5] = bf16_hi(w.z);
            x[6] = bf16_lo(w.w); x[7] = bf16_hi(w.w);
        } else {
            uint4 w0 = *reinterpret_cast<const uint4 *>(v.s + 4 * e0);
            uint4 w1 = *reinterpret_cast<const uint4 *>(v.s + 4 * e0 + 16);
            bad |= nonfinite_f32(w0.x) | nonfinite_f32(w0.y) | nonfinite_f32(w0.z) | nonfinite_f32(w0.w) |
                   nonfinite_f32(w1.x) | nonfinite_f32(w1.y) | nonfinite_f32(w1.z) | nonfinite_f32(w1.w);
            x[0] = __uint_as_float(w0.x); x[1] = __uint_as_float(w0.y);
            x[2] = __uint_as_float(w0.z); x[3] = __uint_as_float(w0.w);
            x[4] = __uint_as_float(w1.x); x[5] = __uint_as_float(w1.y);
            x[6] = __uint_as_float(w1.z); x[7] = __uint_as_float(w1.w);
        }
        return 8;
    }
    if (nv > 8) nv = 8;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if (i < nv) x[i] = ld_one<ES>(v, e0 + i, bad);
    return nv;
}

// Reads one logit straight from global memory.
__device__ __forceinline__ float logit_global(const Params &P, size_t elem) {
    if (P.esize == 2) {
        uint16_t h = __ldg(reinterpret_cast<const unsigned short *>(P.logits) + elem);
        return __uint_as_float(static_cast<uint32_t>(h) << 16);
    }
    return __ldg(reinterpret_cast<const float *>(P.logits) + elem);
}

// ------------------------------------------------------ warp reductions --
__device__ __forceinline__ void argmax_merge(float &v, int &i, float ov, int oi) {
    if (ov > v || (ov == v && oi < i)) {
        v = ov;
        i = oi;
    }
}

__device__ __forceinline__ void warp_argmax(float &v, int &i) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        float ov = __shfl_xor_sync(0xffffffffu, v, off);
        int oi = __shfl_xor_sync(0xffffffffu, i, off);
        argmax_merge(v, i, ov, oi);
    }
}

// Canonical block sum: lane partials combined by an xor butterfly; lane 0's
// value is the block's sum.
__device__ __forceinline__ float warp_butterfly_sum(float s) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, off));
    return s;
}

__device__ __forceinline__ double warp_sum_d(double s) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    return s;
}

__device__ __forceinline__ double warp_incl_scan_d(double s, int lane) {
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        double o = __shfl_up_sync(0xffffffffu, s, off);
        if (lane >= off) s += o;
    }
    return s;
}

// ------------------------------------------------------------ topology --
__device__ __forceinline__ int parent_of(const Params &P, int n) { return P.tree ? P.parent[n] : n - 1; }

__device__ __forceinline__ int node_token(const Params &P, int b, int n) {
    return __ldg(P.tokens + static_cast<size_t>(b) * (P.R - 1) + (n - 1));
}

// Edge parent -> child accepted, given the parent's resolved row state.
__device__ __forceinline__ bool edge_ok(uint32_t rs, bool greedy, int child_token) {
    if (!(rs & kResolved)) return false;
    return greedy ? (static_cast<int>(rs & kIdxMask) == child_token) : ((rs & 1u) != 0u);
}

// ---------------------------------------------------- inverse-CDF search --
// Block weights for the search: residual blocks (bsumB) or exp blocks of one
// row scaled by their chunk's factor 2^((M_c - m) c2).
struct BlockSource {
    const float *bsum;       // nblk block sums of this row
    const Partial *part;     // chunk partials of the row (exp mode), or null
    float m, c2;             // row max and scale (exp mode)
};

__device__ __forceinline__ double chunk_factor(const BlockSource &S, int c) {
    if (!S.part) return 1.0;
    float Mc = __ldcg(&S.part[c].v);
    return static_cast<double>(ex2(__fmul_rn(__fsub_rn(Mc, S.m), S.c2)));
}

__device__ __forceinline__ double block_weight(const BlockSource &S, int beta) {
    double w = static_cast<double>(__ldcg(S.bsum + beta));
    if (S.part) w *= chunk_factor(S, beta / (kChunkA / kBlk));
    return w;
}

// Warp-wide: total weight and the block holding t = u * total.  Returns the
// total; beta/base receive the block and the weight before it (all lanes).
__device__ double locate_block(const BlockSource &S, int nblk, double u, int lane, int &beta, double &base) {
    const int per = (nblk + 31) / 32;
    const int lo = lane * per;
    const int hi = min(nblk, lo + per);
    double s = 0.0;
    for (int i = lo; i < hi; ++i) s += block_weight(S, i);
    double incl = warp_incl_scan_d(s, lane);
    double excl = incl - s;
    double total = __shfl_sync(0xffffffffu, incl, 31);
    double t = u * total;
    unsigned over = __ballot_sync(0xffffffffu, incl > t && hi > lo);
    unsigned nonzero = __ballot_sync(0xffffffffu, s > 0.0);
    int L;
    if (over) L = __ffs(over) - 1;
    else L = nonzero ? 31 - __clz(nonzero) : 0;
    int bsel = -1;
    double bbase = 0.0;
    if (lane == L) {
        double run = excl;
        int last_pos = -1;
        double last_base = excl;
        for (int i = lo; i < hi; ++i) {
            double w = block_weight(S, i);
            if (w > 0.0) {
                last_pos = i;
                last_base = run;
            }
            if (run + w > t && w > 0.0) {
                bsel = i;
                bbase = run;
                break;
            }
            run += w;
        }
        if (bsel < 0) {
            bsel = last_pos >= 0 ? last_pos : lo;
            bbase = last_base;
        }
    }
    beta = __shfl_sync(0xffffffffu, bsel, L);
    base = __shfl_sync(0xffffffffu, bbase, L);
    return total;
}

// Warp-wide scan inside block beta of row (b, row): the first element whose
// running weight exceeds t.  mode 0: exp weights relative to the chunk max,
// scaled by the chunk factor; mode 1: residual weights.
__device__ int scan_block(const Params &P, const BlockSource &S, int b, int row, int beta, double base,
                          double t, int mode, float m, float invS, int lane) {
    const size_t rowz = (static_cast<size_t>(b) * P.R + row) * static_cast<size_t>(P.V);
    const int e0 = beta * kBlk + lane * 8;
    float w[8];
    float s = 0.0f;
    float Mc = 0.0f;
    double fac = 1.0;
    if (mode == 0) {
        int c = beta / (kChunkA / kBlk);
        Mc = __ldcg(&S.part[c].v);
        fac = chunk_factor(S, c);
    }
    const float *qrow = (mode == 1) ? P.q + (static_cast<size_t>(b) * (P.R - 1) + row) * static_cast<size_t>(P.V) : nullptr;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        int e = e0 + i;
        float wi = 0.0f;
        if (e < P.V) {
            float z = logit_global(P, rowz + e);
            wi = (mode == 0) ? w_exp(z, Mc, S.c2) : w_res(z, __ldg(qrow + e), m, S.c2, invS);
        }
        w[i] = wi;
        s = __fadd_rn(s, wi);
    }
    double ls = static_cast<double>(s) * fac;
    double incl = warp_incl_scan_d(ls, lane);
    double lbase = base + (incl - ls);
    unsigned hit = __ballot_sync(0xffffffffu, lbase + ls > t && s > 0.0f);
    unsigned pos = __ballot_sync(0xffffffffu, s > 0.0f);
    int L = hit ? (__ffs(hit) - 1) : (pos ? 31 - __clz(pos) : 0);
    int j = -1;
    if (lane == L) {
        double acc = lbase;
        int last_pos = 0;
        for (int i = 0; i < 8; ++i) {
            if (w[i] > 0.0f) last_pos = i;
            acc += static_cast<double>(w[i]) * fac;
            if (hit && w[i] > 0.0f && acc > t) {
                j = i;
                break;
            }
        }
        if (j < 0) j = last_pos;
        j += e0;
    }
    j = __shfl_sync(0xffffffffu, j, L);
    if (j < 0) j = 0;
    if (j >= P.V) j = P.V - 1;
    return j;
}

// Sample one token from row `row` of request b: residual weights (bsumB) if
// `residual`, else p itself (exp block sums of that row).  Warp-wide.
__device__ int sample_row(const Params &P, int b, int row, bool residual, double u, int lane) {
    RowStat rs;
    rs.m = __ldcg(&P.rowstat[static_cast<size_t>(b) * P.R + row].m);
    rs.S = __ldcg(&P.rowstat[static_cast<size_t>(b) * P.R + row].S);
    const float T = P.temperature[b];
    const float c2 = 1.4426950408889634f / T;
    int beta;
    double base;
    if (residual) {
        BlockSource S{P.bsumB + static_cast<size_t>(b) * P.nblk, nullptr, rs.m, c2};
        double Z = locate_block(S, P.nblk, u, lane, beta, base);
        if (Z > 0.0) {
            float invS = static_cast<float>(1.0 / rs.S);
            return scan_block(P, S, b, row, beta, base, u * Z, 1, rs.m, invS, lane);
        }
        // zero residual mass: sample from p of the same row
    }
    const size_t rowi = static_cast<size_t>(b) * P.R + row;
    BlockSource S{P.bsumA + rowi * P.nblk, P.partial + rowi * P.nca, rs.m, c2};
    double tot = locate_block(S, P.nblk, u, lane, beta, base);
    return scan_block(P, S, b, row, beta, base, u * tot, 0, rs.m, 0.0f, lane);
}

// ------------------------------------------------------- unit decoding --
// Warp 0: decode unit u and decide whether it must be loaded.
__device__ void decode_unit(const Params &P, int u, Unit &U, int lane) {
    U.kind = kEnd;
    if (u < 0 || u >= P.units_total) return;
    if (u < P.units_a) {
        const int per_node = P.B * P.nca;
        int n = u / per_node;
        int rem = u - n * per_node;
        int b = rem / P.nca;
        int c = rem - b * P.nca;
        float T = P.temperature ? __ldg(P.temperature + b) : 0.0f;
        bool greedy = !(T > 0.0f);
        // Is node n already known to be rejected?  Lane i checks the i-th
        // edge on the path from n up to the root.
        bool dead = false;
        if (n > 0) {
            int d = P.tree ? P.depth[n] : n;
            for (int base = 0; base < d && !dead; base += 32) {
                int i = base + lane;
                bool bad = false;
                if (i < d) {
                    int child = n;
                    if (P.tree) {
                        for (int s = 0; s < i; ++s) child = P.parent[child];
                    } else {
                        child = n - i;
                    }
                    int par = parent_of(P, child);
                    uint32_t rs = *reinterpret_cast<volatile const uint32_t *>(P.rowstate + static_cast<size_t>(b) * P.R + par);
                    if (rs & kResolved) bad = !edge_ok(rs, greedy, node_token(P, b, child));
                }
                dead = __any_sync(0xffffffffu, bad);
            }
        }
        U.b = b;
        U.n = n;
        U.c = c;
        U.c2 = greedy ? 0.0f : 1.4426950408889634f / T;
        U.kind = dead ? kASkip : kALoad;
        U.cnt = min(kChunkA, P.V - c * kChunkA);
        size_t elem = (static_cast<size_t>(b) * P.R + n) * static_cast<size_t>(P.V) + static_cast<size_t>(c) * kChunkA;
        U.gz = P.logits + elem * P.esize;
        return;
    }
    const int v = u - P.units_a;
    const int b = v / P.ncb;
    const int c = v - b * P.ncb;
    U.b = b;
    U.c = c;
    U.cnt = min(kChunkB, P.V - c * kChunkB);
    uint32_t st = ld_acquire(P.req_state + b);
    U.kind = kBWait;
    if (st & kDecided) {
        const int a = static_cast<int>(st & kIdxMask);
        if ((st & kNeedsResidual) && a < P.R - 1) {
            U.kind = kBLoad;
            U.n = a;
        } else {
            U.kind = kBSkip;
        }
    }
}

// Thread 0: compute copy geometry for a load unit and issue its bulk copies.
__device__ void issue_unit(const Params &P, Unit &U, uint8_t *stage, uint64_t *bar) {
    auto geom = [](const uint8_t *g, int cnt, int es, unsigned long long end, int &sh, int &tail,
                   const uint8_t *&src, uint32_t &nbytes) {
        unsigned long long a0 = reinterpret_cast<unsigned long long>(g);
        unsigned long long a1 = a0 + static_cast<unsigned long long>(cnt) * es;
        unsigned long long lo = a0 & ~15ull;
        unsigned long long hi = (a1 + 15ull) & ~15ull;
        unsigned long long lim = end & ~15ull;
        if (hi > lim) hi = lim;
        sh = static_cast<int>(a0 - lo);
        if (hi <= lo) {
            nbytes = 0;
            tail = 0;
        } else {
            nbytes = static_cast<uint32_t>(hi - lo);
            long long covered = static_cast<long long>(hi) - static_cast<long long>(a0);
            tail = covered >= static_cast<long long>(cnt) * es ? cnt : static_cast<int>(covered / es);
            if (tail < 0) tail = 0;
        }
        src = reinterpret_cast<const uint8_t *>(lo);
    };
    const uint8_t *srcz;
    uint32_t nz;
    geom(U.gz, U.cnt, P.esize, P.logits_end, U.sh, U.tail, srcz, nz);
    uint32_t nq = 0;
    const uint8_t *srcq = nullptr;
    if (U.kind == kBLoad) {
        geom(U.gq, U.cnt, 4, P.q_end, U.shq, U.tailq, srcq, nq);
    }
    U.bytes = nz + nq;
    if (U.bytes) {
        fence_proxy_async();
        mbar_expect_tx(bar, U.bytes);
        if (nz) bulk_g2s(stage, srcz, nz, bar);
        if (nq) bulk_g2s(stage + kQOff, srcq, nq, bar);
    }
}

// --------------------------------------------------------------- kernel --
template <int ES>
__global__ void __launch_bounds__(kThreads, 4) verify_kernel(const __grid_constant__ Params P) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bar;
    __shared__ Unit s_unit[2];
    __shared__ float s_rv[kWarps];
    __shared__ int s_ri[kWarps];
    __shared__ double s_rd[kWarps];
    __shared__ int s_flag[4];
    __shared__ uint32_t s_rs[kMaxRows];
    __shared__ int s_tok[kMaxRows];
    __shared__ uint8_t s_acc[kMaxRows];

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    uint8_t *stage = smem;
    uint32_t phase = 0;
    uint32_t bad = 0;

    if (tid == 0) {
        mbar_init(&bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // first claim
    if (warp == 0) {
        int u = 0;
        if (lane == 0) u = static_cast<int>(atomicAdd(P.ctrl + 0, 1u));
        u = __shfl_sync(0xffffffffu, u, 0);
        Unit U;
        decode_unit(P, u, U, lane);
        if (lane == 0) s_unit[0] = U;
    }
    __syncthreads();
    int cur = 0;

    while (true) {
        Unit &U = s_unit[cur];
        const int kind0 = U.kind;
        if (kind0 == kEnd) break;
        __syncthreads();   // every thread has read kind0 before thread 0 may rewrite U
        // ---- wait for a B unit's decision (only after all earlier units are done)
        if (kind0 == kBWait) {
            if (tid == 0) {
                unsigned long long t0 = globaltimer();
                uint32_t st = 0;
                while (true) {
                    st = ld_acquire(P.req_state + U.b);
                    if (st & kDecided) break;
                    if (globaltimer() - t0 > kWaitLimitNs) break;
                    __nanosleep(256);
                }
                if (!(st & kDecided)) {
                    set_status(P, SPEC_STATUS_WAIT_TIMEOUT);
                    U.kind = kBSkip;
                } else if ((st & kNeedsResidual) && static_cast<int>(st & kIdxMask) < P.R - 1) {
                    U.kind = kBLoad;
                    U.n = static_cast<int>(st & kIdxMask);
                } else {
                    U.kind = kBSkip;
                }
            }
        }
        // ---- issue the bulk copy
        if (tid == 0 && (U.kind == kALoad || U.kind == kBLoad)) {
            if (U.kind == kBLoad) {
                const size_t ri = static_cast<size_t>(U.b) * P.R + U.n;
                RowStat rs;
                rs.m = __ldcg(&P.rowstat[ri].m);
                rs.S = __ldcg(&P.rowstat[ri].S);
                float T = P.temperature[U.b];
                U.c2 = 1.4426950408889634f / T;
                U.m = rs.m;
                U.invS = static_cast<float>(1.0 / rs.S);
                size_t elem = (static_cast<size_t>(U.b) * P.R + U.n) * static_cast<size_t>(P.V) +
                              static_cast<size_t>(U.c) * kChunkB;
                U.gz = P.logits + elem * P.esize;
                size_t qe = (static_cast<size_t>(U.b) * (P.R - 1) + U.n) * static_cast<size_t>(P.V) +
                            static_cast<size_t>(U.c) * kChunkB;
                U.gq = reinterpret_cast<const uint8_t *>(P.q + qe);
            }
            issue_unit(P, U, stage, &bar);
        }
        __syncthreads();
        // ---- claim and decode the next unit while the copy is in flight
        const int nxt = cur ^ 1;
        if (warp == 0) {
            int u = 0;
            if (lane == 0) u = static_cast<int>(atomicAdd(P.ctrl + 0, 1u));
            u = __shfl_sync(0xffffffffu, u, 0);
            Unit N;
            decode_unit(P, u, N, lane);
            if (lane == 0) s_unit[nxt] = N;
        }
        const int kind = U.kind;
        const int b = U.b, n = U.n, c = U.c;
        // ---- wait for the data
        if ((kind == kALoad || kind == kBLoad) && U.bytes) {
            unsigned long long t0 = 0;
            int spins = 0;
            while (!mbar_try_wait(&bar, phase)) {
                if (++spins == 64) t0 = globaltimer();
                if (spins > 64 && globaltimer() - t0 > kWaitLimitNs) {
                    // The copy never completed: report and stop using this block.
                    set_status(P, SPEC_STATUS_WAIT_TIMEOUT);
                    break;
                }
            }
            phase ^= 1u;
        }
        View vz{stage + U.sh, U.gz, U.cnt, U.tail, U.sh == 0};

        if (kind == kALoad) {
            // ---------------- A unit: argmax (+ softmax statistics) of one chunk
            const int nb = (U.cnt + kBlk - 1) / kBlk;
            float bv = -INFINITY;
            int bi = 0x7fffffff;
            for (int blk = warp; blk < nb; blk += kWarps) {
                float x[8];
                int e0 = blk * kBlk + lane * 8;
                int nv = load8<ES>(vz, e0, x, bad);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (i < nv && x[i] > bv) {
                        bv = x[i];
                        bi = e0 + i;
                    }
            }
            warp_argmax(bv, bi);
            if (lane == 0) {
                s_rv[warp] = bv;
                s_ri[warp] = bi;
            }
            __syncthreads();
            if (warp == 0) {
                float v = lane < kWarps ? s_rv[lane] : -INFINITY;
                int i = lane < kWarps ? s_ri[lane] : 0x7fffffff;
                warp_argmax(v, i);
                if (lane == 0) {
                    s_rv[0] = v;
                    s_ri[0] = i;
                }
            }
            __syncthreads();
            const float M = s_rv[0];
            const int Mi = s_ri[0];
            double csum = 0.0;
            if (U.c2 != 0.0f) {
                // sampled: 256-element block sums of exp2((z - M) c2)
                float *bs = P.bsumA + (static_cast<size_t>(b) * P.R + n) * P.nblk + static_cast<size_t>(c) * (kChunkA / kBlk);
                double wsum = 0.0;
                for (int blk = warp; blk < nb; blk += kWarps) {
                    float x[8];
                    int e0 = blk * kBlk + lane * 8;
                    int nv = load8<ES>(vz, e0, x, bad);
                    float s = 0.0f;
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        if (i < nv) s = __fadd_rn(s, w_exp(x[i], M, U.c2));
                    s = warp_butterfly_sum(s);
                    if (lane == 0) {
                        bs[blk] = s;
                        wsum += static_cast<double>(s);
                    }
                }
                if (lane == 0) s_rd[warp] = wsum;
                __syncthreads();
                if (tid == 0)
                    for (int w = 0; w < kWarps; ++w) csum += s_rd[w];
            }
            // ---- publish the partial; the last chunk of the row resolves it
            __threadfence();
            __syncthreads();
            if (tid == 0) {
                const size_t ri = static_cast<size_t>(b) * P.R + n;
                Partial pr;
                pr.v = M;
                pr.idx = (Mi == 0x7fffffff) ? c * kChunkA : c * kChunkA + Mi;
                pr.s = csum;
                P.partial[ri * P.nca + c] = pr;
                uint32_t old = atom_add_acqrel(P.row_done + ri, 1u);
                s_flag[0] = (old == static_cast<uint32_t>(P.nca - 1));
                atomicAdd(P.stats + 0, 1ull);
                atomicAdd(P.stats + 4, static_cast<unsigned long long>(U.bytes));
            }
            __syncthreads();
            if (s_flag[0] && warp == 0) {
                // ---------------- row resolution (one warp)
                const size_t ri = static_cast<size_t>(b) * P.R + n;
                const Partial *pp = P.partial + ri * P.nca;
                uint32_t rsv;
                if (U.c2 == 0.0f) {
                    float v = -INFINITY;
                    int i = 0x7fffffff;
                    for (int q = lane; q < P.nca; q += 32) argmax_merge(v, i, __ldcg(&pp[q].v), __ldcg(&pp[q].idx));
                    warp_argmax(v, i);
                    if (i < 0 || i >= P.V) i = 0;
                    rsv = kResolved | static_cast<uint32_t>(i);
                } else {
                    float m = -INFINITY;
                    for (int q = lane; q < P.nca; q += 32) m = fmaxf(m, __ldcg(&pp[q].v));
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
                    double S = 0.0;
                    for (int q = lane; q < P.nca; q += 32) {
                        float Mc = __ldcg(&pp[q].v);
                        S += __ldcg(&pp[q].s) * static_cast<double>(ex2(__fmul_rn(__fsub_rn(Mc, m), U.c2)));
                    }
                    S = warp_sum_d(S);
                    uint32_t acc = 0;
                    if (lane == 0) {
                        RowStat st;
                        st.m = m;
                        st.pad = 0.0f;
                        st.S = S;
                        P.rowstat[ri] = st;
                        if (n < P.R - 1) {
                            // accept test of the draft token checked by this row
                            int x = node_token(P, b, n + 1);
                            if (x < 0 || x >= P.V) {
                                set_status(P, SPEC_STATUS_TOKEN_RANGE);
                            } else {
                                float zx = logit_global(P, ri * P.V + x);
                                double ph = static_cast<double>(ex2(__fmul_rn(__fsub_rn(zx, m), U.c2))) / S;
                                float qh = __ldg(P.q + (static_cast<size_t>(b) * (P.R - 1) + n) * P.V + x);
                                if (qh == 0.0f) {
                                    acc = 1;
                                } else {
                                    double ua = static_cast<double>(__ldg(P.u_accept + static_cast<size_t>(b) * (P.R - 1) + n));
                                    acc = ua < ph / static_cast<double>(qh);
                                }
                            }
                        }
                    }
                    rsv = kResolved | __shfl_sync(0xffffffffu, acc, 0);
                }
                if (lane == 0) {
                    __threadfence();
                    st_release(P.rowstate + ri, rsv);
                }
            }
        } else if (kind == kBLoad) {
            // ---------------- B unit: residual block sums of one chunk of row a
            View vq{stage + kQOff + U.shq, U.gq, U.cnt, U.tailq, U.shq == 0};
            const int nb = (U.cnt + kBlk - 1) / kBlk;
            float *bs = P.bsumB + static_cast<size_t>(b) * P.nblk + static_cast<size_t>(c) * (kChunkB / kBlk);
            uint32_t qbad = 0;
            for (int blk = warp; blk < nb; blk += kWarps) {
                float x[8], y[8];
                int e0 = blk * kBlk + lane * 8;
                int nv = load8<ES>(vz, e0, x, bad);
                load8<4>(vq, e0, y, qbad);
                float s = 0.0f;
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (i < nv) s = __fadd_rn(s, w_res(x[i], y[i], U.m, U.c2, U.invS));
                s = warp_butterfly_sum(s);
                if (lane == 0) bs[blk] = s;
            }
            __threadfence();
            __syncthreads();
            if (tid == 0) {
                uint32_t old = atom_add_acqrel(P.res_done + b, 1u);
                s_flag[0] = (old == static_cast<uint32_t>(P.ncb - 1));
                atomicAdd(P.stats + 2, 1ull);
                atomicAdd(P.stats + 4, static_cast<unsigned long long>(U.bytes));
            }
            __syncthreads();
            if (s_flag[0] && warp == 0) {
                // ---------------- residual sample of request b at row a (one warp)
                __threadfence();
                const int a = U.n;
                double u = static_cast<double>(__ldg(P.u_sample + static_cast<size_t>(b) * P.R + a));
                int tok = sample_row(P, b, a, true, u, lane);
                if (lane == 0) P.out_tokens[static_cast<size_t>(b) * (P.D + 1) + a] = tok;
            }
        } else if (kind == kASkip) {
            if (tid == 0) atomicAdd(P.stats + 1, 1ull);
        } else if (kind == kBSkip) {
            if (tid == 0) atomicAdd(P.stats + 3, 1ull);
        }

        // ---- request completion (A units only, loaded or skipped)
        if (kind == kALoad || kind == kASkip) {
            __syncthreads();
            if (tid == 0) {
                __threadfence();
                uint32_t old = atom_add_acqrel(P.req_done + b, 1u);
                s_flag[1] = (old == static_cast<uint32_t>(P.R * P.nca - 1));
            }
            __syncthreads();
            if (s_flag[1]) {
                // ---------------- finalize request b
                __threadfence();
                int range_bad = 0;
                for (int i = tid; i < P.R; i += kThreads) {
                    s_rs[i] = *reinterpret_cast<volatile const uint32_t *>(P.rowstate + static_cast<size_t>(b) * P.R + i);
                    s_tok[i] = i > 0 ? node_token(P, b, i) : -1;
                    if (i > 0 && (s_tok[i] < 0 || s_tok[i] >= P.V)) range_bad = 1;
                }
                if (__any_sync(0xffffffffu, range_bad) && lane == 0) set_status(P, SPEC_STATUS_TOKEN_RANGE);
                __syncthreads();
                if (tid == 0) {
                    const float T = P.temperature ? P.temperature[b] : 0.0f;
                    const bool greedy = !(T > 0.0f);
                    s_acc[0] = 1;
                    int best = 0;
                    for (int i = 1; i < P.R; ++i) {
                        int p = parent_of(P, i);
                        bool ok = s_acc[p] && edge_ok(s_rs[p], greedy, s_tok[i]);
                        s_acc[i] = ok;
                        int di = P.tree ? P.depth[i] : i;
                        int db = P.tree ? P.depth[best] : best;
                        if (ok && di > db) best = i;
                    }
                    const int d = P.tree ? P.depth[best] : best;
                    int32_t *ot = P.out_tokens + static_cast<size_t>(b) * (P.D + 1);
                    // path (root first) into s_ri as scratch-free walk
                    int node = best;
                    for (int i = d; i >= 1; --i) {
                        ot[i - 1] = s_tok[node];
                        if (P.out_path) P.out_path[static_cast<size_t>(b) * (P.D + 1) + i] = node;
                        node = parent_of(P, node);
                    }
                    if (P.out_path) {
                        P.out_path[static_cast<size_t>(b) * (P.D + 1)] = 0;
                        for (int i = d + 1; i <= P.D; ++i) P.out_path[static_cast<size_t>(b) * (P.D + 1) + i] = -1;
                    }
                    for (int i = d + 1; i <= P.D; ++i) ot[i] = -1;
                    uint32_t st = kDecided;
                    if (greedy) {
                        uint32_t rs = s_rs[best];
                        ot[d] = (rs & kResolved) ? static_cast<int>(rs & kIdxMask) : 0;
                    } else if (d < P.R - 1) {
                        st |= kNeedsResidual | static_cast<uint32_t>(d);
                        ot[d] = -1;   // written by the residual pass
                    }
                    P.out_count[b] = P.tree ? d + 1 : d;
                    s_flag[2] = (!greedy && d == P.R - 1) ? 1 : 0;
                    s_flag[3] = static_cast<int>(st);
                }
                __syncthreads();
                if (s_flag[2] && warp == 0) {
                    // bonus token: every draft accepted, sample from p at the last row
                    const int a = P.R - 1;
                    double u = static_cast<double>(__ldg(P.u_sample + static_cast<size_t>(b) * P.R + a));
                    int tok = sample_row(P, b, a, false, u, lane);
                    if (lane == 0) P.out_tokens[static_cast<size_t>(b) * (P.D + 1) + a] = tok;
                }
                if (tid == 0) {
                    __threadfence();
                    st_release(P.req_state + b, static_cast<uint32_t>(s_flag[3]));
                }
            }
        }
        __syncthreads();
        cur = nxt;
    }

    // ---- report data problems, then the last block out clears the counters
    bad = __any_sync(0xffffffffu, bad != 0);
    if (lane == 0 && bad) set_status(P, SPEC_STATUS_NONFINITE);
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        uint32_t old = atom_add_acqrel(P.ctrl + 1, 1u);
        s_flag[0] = (old == gridDim.x - 1);
    }
    __syncthreads();
    if (s_flag[0]) {
        __threadfence();
        for (uint32_t i = tid; i < P.reset_words; i += kThreads) P.reset_base[i] = 0u;
        __threadfence();
    }
}

// ------------------------------------------------------------ slot fix-up --
__global__ void fixup_kernel(int64_t *slots, int B, int P, const int32_t *num_acc, const int32_t *path,
                             int stride, int64_t pad) {
    const long long total = static_cast<long long>(B) * P;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int b = static_cast<int>(idx / P);
        const int j = static_cast<int>(idx - static_cast<long long>(b) * P);
        bool keep;
        if (!path) {
            keep = j <= __ldg(num_acc + b);
        } else {
            keep = (j == 0);
            const int32_t *pb = path + static_cast<size_t>(b) * stride;
            for (int i = 0; i < stride && !keep; ++i) keep = (__ldg(pb + i) == j);
        }
        if (!keep) slots[idx] = pad;
    }
}

// =================================================================== host ==
thread_local char g_err[512] = "";

spec_status_t fail(spec_status_t s, const char *fmt, const char *detail = "") {
    snprintf(g_err, sizeof g_err, fmt, detail);
    return s;
}

struct Layout {
    size_t stats, reset, reset_bytes, ctrl, row_done, rowstate, req_done, req_state, res_done;
    size_t rowstat, partial, bsumA, bsumB, total;
    int nca, ncb, nblk;
};

size_t up256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

bool make_layout(int B, int R, int V, Layout &L) {
    if (B < 1 || R < 1 || R > kMaxRows || V < 1 || V >= (1 << 30)) return false;
    L.nca = (V + kChunkA - 1) / kChunkA;
    L.ncb = (V + kChunkB - 1) / kChunkB;
    L.nblk = (V + kBlk - 1) / kBlk;
    const size_t BR = static_cast<size_t>(B) * R;
    size_t off = 0;
    L.stats = off;
    off = up256(off + 64);
    L.reset = off;
    L.ctrl = off;
    off += 32 * 4;
    L.row_done = off;
    off += BR * 4;
    L.rowstate = off;
    off += BR * 4;
    L.req_done = off;
    off += static_cast<size_t>(B) * 4;
    L.req_state = off;
    off += static_cast<size_t>(B) * 4;
    L.res_done = off;
    off += static_cast<size_t>(B) * 4;
    off = up256(off);
    L.reset_bytes = off - L.reset;
    L.rowstat = off;
    off = up256(off + BR * sizeof(RowStat));
    L.partial = off;
    off = up256(off + BR * L.nca * sizeof(Partial));
    L.bsumA = off;
    off = up256(off + BR * L.nblk * 4);
    L.bsumB = off;
    off = up256(off + static_cast<size_t>(B) * L.nblk * 4);
    L.total = off;
    return true;
}

struct DeviceInfo {
    int sms = 0;
    int ok = 0;
    int blocks_per_sm[2] = {0, 0};
    uint8_t *noalloc_scratch = nullptr;   // device address of g_noalloc_scratch on this device
};

std::mutex g_mu;
DeviceInfo g_dev[64];

spec_status_t device_info(DeviceInfo *&out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return fail(SPEC_ERR_UNSUPPORTED, "device index out of range%s");
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo &D = g_dev[dev];
    if (!D.ok) {
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (major != 10 || minor != 3) {
            char buf[64];
            snprintf(buf, sizeof buf, "%d.%d", major, minor);
            return fail(SPEC_ERR_UNSUPPORTED, "needs compute capability 10.3 (sm_103a), device is %s", buf);
        }
        cudaDeviceGetAttribute(&D.sms, cudaDevAttrMultiProcessorCount, dev);
        e = cudaFuncSetAttribute(verify_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kStageBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(verify_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, kStageBytes);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&D.blocks_per_sm[0], verify_kernel<2>, kThreads, kStageBytes);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&D.blocks_per_sm[1], verify_kernel<4>, kThreads, kStageBytes);
        if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "kernel setup: %s", cudaGetErrorString(e));
        D.ok = 1;
    }
    out = &D;
    return SPEC_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

spec_status_t launch_verify(Params &P, spec_dtype_t dtype, void *workspace, size_t ws_bytes, void *stream) {
    Layout L;
    if (!make_layout(P.B, P.R, P.V, L)) return fail(SPEC_ERR_INVALID_ARG, "invalid sizes%s");
    if (!workspace || ws_bytes < L.total)
        return fail(SPEC_ERR_INVALID_ARG, "workspace missing or smaller than spec_workspace_bytes()%s");
    if (!aligned16(workspace)) return fail(SPEC_ERR_INVALID_ARG, "workspace must be 16-byte aligned%s");
    DeviceInfo *D = nullptr;
    spec_status_t s = device_info(D);
    if (s != SPEC_OK) return s;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    P.stats = reinterpret_cast<unsigned long long *>(ws + L.stats);
    P.ctrl = reinterpret_cast<uint32_t *>(ws + L.ctrl);
    P.row_done = reinterpret_cast<uint32_t *>(ws + L.row_done);
    P.rowstate = reinterpret_cast<uint32_t *>(ws + L.rowstate);
    P.req_done = reinterpret_cast<uint32_t *>(ws + L.req_done);
    P.req_state = reinterpret_cast<uint32_t *>(ws + L.req_state);
    P.res_done = reinterpret_cast<uint32_t *>(ws + L.res_done);
    P.reset_base = reinterpret_cast<uint32_t *>(ws + L.reset);
    P.reset_words = static_cast<uint32_t>(L.reset_bytes / 4);
    P.rowstat = reinterpret_cast<RowStat *>(ws + L.rowstat);
    P.partial = reinterpret_cast<Partial *>(ws + L.partial);
    P.bsumA = reinterpret_cast<float *>(ws + L.bsumA);
    P.bsumB = reinterpret_cast<float *>(ws + L.bsumB);
    P.esize = dtype == SPEC_BF16 ? 2 : 4;
    P.nca = L.nca;
    P.ncb = L.ncb;
    P.nblk = L.nblk;
    const long long ua = static_cast<long long>(P.B) * P.R * L.nca;
    const long long ub = P.q ? static_cast<long long>(P.B) * L.ncb : 0;
    if (ua + ub >= (1ll << 31) - 1024) return fail(SPEC_ERR_INVALID_ARG, "batch too large%s");
    P.units_a = static_cast<int>(ua);
    P.units_total = static_cast<int>(ua + ub);
    const size_t zbytes = static_cast<size_t>(P.B) * P.R * static_cast<size_t>(P.V) * P.esize;
    P.logits_end = reinterpret_cast<unsigned long long>(P.logits) + zbytes;
    P.q_end = P.q ? reinterpret_cast<unsigned long long>(P.q) + static_cast<size_t>(P.B) * (P.R - 1) * static_cast<size_t>(P.V) * 4 : 0;
    const int per_sm = D->blocks_per_sm[dtype == SPEC_BF16 ? 0 : 1];
    long long grid = static_cast<long long>(D->sms) * (per_sm > 0 ? per_sm : 1);
    if (grid > P.units_total) grid = P.units_total;
    if (grid < 1) grid = 1;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dtype == SPEC_BF16)
        verify_kernel<2><<<static_cast<unsigned>(grid), kThreads, kStageBytes, st>>>(P);
    else
        verify_kernel<4><<<static_cast<unsigned>(grid), kThreads, kStageBytes, st>>>(P);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "verify launch: %s", cudaGetErrorString(e));
    return SPEC_OK;
}

// ------------------------------------------------------ no-alloc scratch --
// Scratch of spec_verify_chain_noalloc: a fixed device array that exists on
// every GPU on which the library's module is loaded, until the process exits.
constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(16) << 20;   // 16 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Host code may not use g_noalloc_scratch's name as a pointer (it is a host-side
// stand-in); the device address is looked up once per device, with that
// device current, and cached.
spec_status_t noalloc_scratch_ptr(uint8_t *&out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return fail(SPEC_ERR_UNSUPPORTED, "device index out of range%s");
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo &D = g_dev[dev];
    if (!D.noalloc_scratch) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p)
            return fail(SPEC_ERR_CUDA, "cudaGetSymbolAddress(no-alloc scratch): %s", cudaGetErrorString(e));
        D.noalloc_scratch = static_cast<uint8_t *>(p);
    }
    out = D.noalloc_scratch;
    return SPEC_OK;
}

}  // namespace sv

// =============================================================== C ABI ==
using namespace sv;

extern "C" size_t spec_workspace_bytes(int B, int rows, int V, spec_dtype_t dtype) {
    (void)dtype;
    Layout L;
    if (!make_layout(B, rows, V, L)) return 0;
    return L.total;
}

extern "C" spec_status_t spec_workspace_init(void *workspace, size_t bytes, void *stream) {
    if (!workspace) return fail(SPEC_ERR_INVALID_ARG, "workspace is NULL%s");
    cudaError_t e = cudaMemsetAsync(workspace, 0, bytes, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "cudaMemsetAsync: %s", cudaGetErrorString(e));
    return SPEC_OK;
}

extern "C" spec_status_t spec_verify_chain(const void *target_logits, spec_dtype_t dtype, const float *draft_probs,
                                           const int32_t *draft_tokens, const float *temperature,
                                           const float *u_accept, const float *u_sample, int B, int k, int V,
                                           int32_t *out_tokens, int32_t *out_num_accepted, int32_t *d_status,
                                           void *workspace, size_t workspace_bytes, void *stream) {
    g_err[0] = 0;
    if (dtype != SPEC_BF16 && dtype != SPEC_FP32) return fail(SPEC_ERR_INVALID_ARG, "unknown dtype%s");
    if (B < 1 || k < 1 || k > kMaxRows - 1 || V < 1 || V >= (1 << 30))
        return fail(SPEC_ERR_INVALID_ARG, "sizes out of range (1<=B, 1<=k<=255, 1<=V<2^30)%s");
    if (!target_logits || !draft_tokens || !out_tokens || !out_num_accepted)
        return fail(SPEC_ERR_INVALID_ARG, "a required pointer is NULL%s");
    const bool sampled = draft_probs || u_accept || u_sample || temperature;
    if (sampled && (!draft_probs || !u_accept || !u_sample || !temperature))
        return fail(SPEC_ERR_INVALID_ARG,
                    "draft_probs, temperature, u_accept and u_sample must be all given or all NULL%s");
    if (!aligned16(target_logits) || (draft_probs && !aligned16(draft_probs)))
        return fail(SPEC_ERR_INVALID_ARG, "target_logits and draft_probs must be 16-byte aligned%s");
    Params P;
    memset(&P, 0, sizeof P);
    P.logits = static_cast<const uint8_t *>(target_logits);
    P.q = draft_probs;
    P.tokens = draft_tokens;
    P.temperature = temperature;
    P.u_accept = u_accept;
    P.u_sample = u_sample;
    P.out_tokens = out_tokens;
    P.out_count = out_num_accepted;
    P.out_path = nullptr;
    P.status = d_status;
    P.B = B;
    P.R = k + 1;
    P.V = V;
    P.D = k;
    P.tree = 0;
    return launch_verify(P, dtype, workspace, workspace_bytes, stream);
}

extern "C" spec_status_t spec_verify_tree(const void *target_logits, spec_dtype_t dtype, const int32_t *node_tokens,
                                          const int32_t *parent, int B, int N, int V, int max_depth,
                                          int32_t *out_path, int32_t *out_tokens, int32_t *out_len,
                                          int32_t *d_status, void *workspace, size_t workspace_bytes,
                                          void *stream) {
    g_err[0] = 0;
    if (dtype != SPEC_BF16 && dtype != SPEC_FP32) return fail(SPEC_ERR_INVALID_ARG, "unknown dtype%s");
    if (B < 1 || N < 0 || N > kMaxRows - 1 || V < 1 || V >= (1 << 30) || max_depth < 0)
        return fail(SPEC_ERR_INVALID_ARG, "sizes out of range (1<=B, 0<=N<=255, 1<=V<2^30)%s");
    if (!target_logits || !parent || !out_path || !out_tokens || !out_len || (N > 0 && !node_tokens))
        return fail(SPEC_ERR_INVALID_ARG, "a required pointer is NULL%s");
    if (!aligned16(target_logits)) return fail(SPEC_ERR_INVALID_ARG, "target_logits must be 16-byte aligned%s");
    Params P;
    memset(&P, 0, sizeof P);
    if (parent[0] != -1) return fail(SPEC_ERR_INVALID_ARG, "parent[0] must be -1%s");
    P.parent[0] = -1;
    P.depth[0] = 0;
    int maxd = 0;
    for (int n = 1; n <= N; ++n) {
        if (parent[n] < 0 || parent[n] >= n) return fail(SPEC_ERR_INVALID_ARG, "parent[n] must satisfy 0 <= parent[n] < n%s");
        P.parent[n] = static_cast<int16_t>(parent[n]);
        P.depth[n] = static_cast<uint8_t>(P.depth[parent[n]] + 1);
        if (P.depth[n] > maxd) maxd = P.depth[n];
    }
    if (max_depth < maxd) return fail(SPEC_ERR_INVALID_ARG, "max_depth is smaller than the tree depth%s");
    P.logits = static_cast<const uint8_t *>(target_logits);
    P.q = nullptr;
    P.tokens = node_tokens;
    P.temperature = nullptr;
    P.out_tokens = out_tokens;
    P.out_count = out_len;
    P.out_path = out_path;
    P.status = d_status;
    P.B = B;
    P.R = N + 1;
    P.V = V;
    P.D = max_depth;
    P.tree = 1;
    return launch_verify(P, dtype, workspace, workspace_bytes, stream);
}

extern "C" spec_status_t spec_fixup_slots(int64_t *slot_mapping, int B, int P, const int32_t *num_accepted,
                                          const int32_t *path, int path_stride, int64_t padding_slot_id,
                                          void *stream) {
    g_err[0] = 0;
    if (B < 0 || P < 0) return fail(SPEC_ERR_INVALID_ARG, "negative size%s");
    if (B == 0 || P == 0) return SPEC_OK;
    if (!slot_mapping) return fail(SPEC_ERR_INVALID_ARG, "slot_mapping is NULL%s");
    if (!path && !num_accepted) return fail(SPEC_ERR_INVALID_ARG, "need num_accepted (chain) or path (tree)%s");
    if (path && path_stride < 1) return fail(SPEC_ERR_INVALID_ARG, "path_stride must be >= 1%s");
    const long long total = static_cast<long long>(B) * P;
    long long blocks = (total + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    fixup_kernel<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        slot_mapping, B, P, num_accepted, path, path_stride, padding_slot_id);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "fixup launch: %s", cudaGetErrorString(e));
    return SPEC_OK;
}

extern "C" spec_status_t spec_tree_from_choices(const int32_t *flat, const int32_t *lens, int n, int32_t *parent,
                                                int32_t *cu_per_level, int32_t *child_per_level, int *depth) {
    g_err[0] = 0;
    if (n < 1 || n > kMaxRows - 1 || !flat || !lens || !parent || !depth)
        return fail(SPEC_ERR_INVALID_ARG, "need 1 <= n <= 255 tuples and non-NULL arrays%s");
    int offs[kMaxRows];
    int off = 0;
    for (int i = 0; i < n; ++i) {
        if (lens[i] < 1 || lens[i] > kMaxRows) return fail(SPEC_ERR_INVALID_ARG, "tuple length out of range%s");
        if (i > 0 && lens[i] < lens[i - 1]) return fail(SPEC_ERR_INVALID_ARG, "tree_choices must be in level order%s");
        offs[i] = off;
        off += lens[i];
    }
    const int D = lens[n - 1];
    int counts[kMaxRows];
    for (int l = 0; l < D; ++l) counts[l] = 0;
    parent[0] = -1;
    for (int i = 0; i < n; ++i) {
        counts[lens[i] - 1]++;
        if (lens[i] == 1) {
            parent[i + 1] = 0;
            continue;
        }
        int found = -1;
        for (int j = 0; j < i && found < 0; ++j) {
            if (lens[j] != lens[i] - 1) continue;
            bool same = true;
            for (int t = 0; t < lens[j] && same; ++t) same = flat[offs[j] + t] == flat[offs[i] + t];
            if (same) found = j;
        }
        if (found < 0) return fail(SPEC_ERR_INVALID_ARG, "a tuple's prefix is missing or comes later%s");
        parent[i + 1] = found + 1;
    }
    for (int l = 0; l < D; ++l)
        if (counts[l] == 0) return fail(SPEC_ERR_INVALID_ARG, "a level has no nodes%s");
    if (cu_per_level) {
        int acc = 0;
        for (int l = 0; l < D; ++l) cu_per_level[l] = (acc += counts[l]);
    }
    if (child_per_level) {
        child_per_level[0] = counts[0];
        for (int l = 1; l < D; ++l) child_per_level[l] = counts[l] / counts[l - 1];
    }
    *depth = D;
    return SPEC_OK;
}

extern "C" const char *spec_last_error(void) { return g_err; }

extern "C" size_t spec_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

extern "C" spec_status_t spec_verify_chain_noalloc(const void *target_logits, spec_dtype_t dtype,
                                                   const float *draft_probs, const int32_t *draft_tokens,
                                                   const float *temperature, const float *u_accept,
                                                   const float *u_sample, int B, int k, int V,
                                                   int32_t *out_tokens, int32_t *out_num_accepted,
                                                   int32_t *d_status, void *stream) {
    g_err[0] = 0;
    if (dtype != SPEC_BF16 && dtype != SPEC_FP32) return fail(SPEC_ERR_INVALID_ARG, "unknown dtype%s");
    if (B < 1 || k < 1 || k > kMaxRows - 1 || V < 1 || V >= (1 << 30))
        return fail(SPEC_ERR_INVALID_ARG, "sizes out of range (1<=B, 1<=k<=255, 1<=V<2^30)%s");
    if (!target_logits || !draft_tokens || !out_tokens || !out_num_accepted)
        return fail(SPEC_ERR_INVALID_ARG, "a required pointer is NULL%s");
    const bool sampled = draft_probs || u_accept || u_sample || temperature;
    if (sampled && (!draft_probs || !u_accept || !u_sample || !temperature))
        return fail(SPEC_ERR_INVALID_ARG,
                    "draft_probs, temperature, u_accept and u_sample must be all given or all NULL%s");
    if (!aligned16(target_logits) || (draft_probs && !aligned16(draft_probs)))
        return fail(SPEC_ERR_INVALID_ARG, "target_logits and draft_probs must be 16-byte aligned%s");
    Layout L;
    if (!make_layout(B, k + 1, V, L)) return fail(SPEC_ERR_INVALID_ARG, "invalid sizes%s");
    if (L.total > kNoAllocScratchBytes) {
        char buf[160];
        snprintf(buf, sizeof buf, "these sizes need %zu bytes of scratch; the static scratch holds %zu bytes",
                 L.total, kNoAllocScratchBytes);
        return fail(SPEC_ERR_INVALID_ARG, "%s (use spec_verify_chain with a workspace)", buf);
    }
    uint8_t *scratch = nullptr;
    spec_status_t s = noalloc_scratch_ptr(scratch);
    if (s != SPEC_OK) return s;
    // The scratch keeps whatever the previous call left; only this layout's
    // counter region has to start at zero.
    cudaError_t e = cudaMemsetAsync(scratch + L.reset, 0, L.reset_bytes, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "clearing the no-alloc scratch: %s", cudaGetErrorString(e));
    Params P;
    memset(&P, 0, sizeof P);
    P.logits = static_cast<const uint8_t *>(target_logits);
    P.q = draft_probs;
    P.tokens = draft_tokens;
    P.temperature = temperature;
    P.u_accept = u_accept;
    P.u_sample = u_sample;
    P.out_tokens = out_tokens;
    P.out_count = out_num_accepted;
    P.out_path = nullptr;
    P.status = d_status;
    P.B = B;
    P.R = k + 1;
    P.V = V;
    P.D = k;
    P.tree = 0;
    return launch_verify(P, dtype, scratch, kNoAllocScratchBytes, stream);
}
