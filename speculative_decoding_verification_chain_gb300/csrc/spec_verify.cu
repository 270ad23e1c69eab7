// spec_verify.cu -- GB300 (sm_103a) verify-and-accept for speculative decoding.
//
// One persistent kernel (one block per SM) verifies chains (greedy or sampled,
// per request) and greedy token trees.  A chain is handled as a tree whose
// node n has parent n-1, so both share one scheduler.  The host part of this
// file holds the entry points and routes each call: sampled padded chains
// whose per-request clusters all fit on the GPU go to chain_cluster.cu, greedy
// trees of at most 64 rows and small greedy padded chains to
// greedy_cluster.cu, the rest to this kernel.
//
// Work.  A row of logits is cut into stages of at most 64 KiB (32768 bf16 or
// 16384 fp32 elements), balanced in size and a whole number of 256-element
// blocks.  An "A unit" is one split of one row: the whole row, or a run of its
// stages when the batch has too few rows to fill the GPU.  A "B unit" is a
// 12288-element chunk (four stages of 3072 elements, logits plus q) of the
// rejected row of a sampled request: the residual pass.  Units are numbered
// (node, request, split)-major, so a parent row is claimed long before its
// children; B units come after every A unit.
//
// Roles inside a block (480 threads):
//   * warp 0, producer: claims units with one global atomic (one claim ahead),
//     drops a row whose node is already known to be rejected (an ancestor
//     edge resolved and failed) without reading it, and streams the rest into
//     a ring of three shared-memory stages, one cp.async.bulk copy each,
//     completing on per-stage mbarriers;
//   * warps 3..14, consumers: reduce each stage in 24 KiB passes -- running
//     argmax (greedy) or, per 256-element block, the block max M and
//     sum 2^((z - M) log2(e)/T) (sampled), or the residual block sums of
//     max(0, p - q) (B units) -- and hand each finished unit to an epilogue;
//   * warps 1..2, epilogues: combine a unit's partials; the last split of a
//     row resolves it (its argmax, or its softmax statistics and the accept
//     test min(1, p/q) of its one child).  Each resolved row is recorded in
//     its request's 64-bit mask of resolved rows (requests over 64 rows count
//     settled rows instead); the row that decides the request -- a chain
//     whose resolved prefix holds a rejection, or a tree whose accepted
//     nodes are all resolved -- walks the tree, picks the deepest accepted
//     node, writes the outputs and (chains, when asked) pads the rejected
//     slots of slot_mapping.  A sampled request
//     rejected at row a publishes that decision as soon as row a resolves; its
//     B units then run, and the last one locates u * (residual mass) in the
//     block sums and scans one 256-element block for the token.  The residual
//     is never written out.
//
// Every wait is bounded by a wall-clock limit and reports
// SPEC_STATUS_WAIT_TIMEOUT instead of hanging.  The last block to exit clears
// the workspace counters, so the next call (or graph replay) starts clean.
//
// Arithmetic: logits are widened to fp32 exactly; exponentials use the SFU
// ex2 approximation on (z - M) * log2(e)/T with M a block max; row statistics
// and the inverse-CDF prefixes across blocks are two-float fp32 sums (about
// 44 significant bits) rather than fp64, whose issue rate on this part is low.

#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "common.h"
#include "ptx.cuh"
#include "twofloat.cuh"
#include "spec_verify.h"

namespace sv {

// ---------------------------------------------------------------- config --
constexpr int kConsumerWarps = 12;
constexpr int kConsumerLanes = 32 * kConsumerWarps;
constexpr int kEpilogueWarps = 2;
constexpr int kThreads = 32 * (1 + kEpilogueWarps + kConsumerWarps);   // producer, epilogues, consumers
// The bulk-copy engine of an SM completes about one copy at a time, so the
// per-SM stream rate grows with the copy size: three 64 KiB stages, each one
// copy, consumed in passes of 24 KiB (the consumers' register tiles).
constexpr int kStages = 3;
constexpr int kSubBytes = 65536;                       // data bytes per stage (at most)
constexpr int kPassBytes = 24576;                      // bytes per consumer pass
constexpr int kStageBytes = kSubBytes + 128;
constexpr int kSubPerB = 4;                             // B stages per B unit
constexpr int kResSlots = 4;
constexpr int kBlk = 256;                               // canonical block: 32 lanes x 8 elements
constexpr int kMaxRows = SPEC_MAX_ROWS;
constexpr uint32_t kResolved = 0x80000000u;
constexpr uint32_t kIdxMask = 0x3fffffffu;
constexpr uint32_t kDecided = 0x80000000u;
constexpr uint32_t kNeedsResidual = 0x40000000u;
constexpr unsigned long long kWaitLimitNs = 500000000ull;   // 0.5 s: default wait limit; always the limit
                                                            // on copies still in flight at exit
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kEarlyMax = 4;                            // children per node given an early-rejection check
constexpr uint32_t kFirstF = 1u << 6;                   // stage flag: first stage of its unit
constexpr int kThrOff = kSubBytes + 64;                 // A stage: 16-byte chunks holding the children's logits
static_assert(kThrOff + 16 * kEarlyMax <= kStageBytes, "threshold chunks do not fit in the stage");
static_assert(kResSlots % kEpilogueWarps == 0, "result slots must split evenly over the epilogue warps");

enum Kind : int { kEnd = 0, kA = 1, kB = 2 };

struct RowStat {
    float m;        // row max of raw logits
    float Sh, Sl;   // sum_j 2^((z_j - m) * c2), two-float
    float pad;
};

struct __align__(16) Partial {  // result of one split of a row (read as one float4)
    float v;      // greedy: max value; sampled: max logit m
    int32_t idx;  // greedy: row index of the first occurrence of v
    float sh, sl; // sampled: sum of 2^((z - m) c2) over the split, two-float
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
    int64_t *slots;              // chains: slot_mapping fixed up in the finalisation, or null
    int64_t pad;                 // ... PADDING_SLOT_ID
    // workspace
    unsigned long long *stats;   // [8], never cleared by the kernel
    uint32_t *ctrl;              // [32]: 0 claim counter, 1 exit counter
    uint32_t *row_ctr;           // [B*R] split arrival counters
    uint32_t *rowstate;          // [B*R]
    uint32_t *req_ctr;           // [B] settled rows
    uint32_t *req_state;         // [B] decision
    uint32_t *res_ctr;           // [B] residual units done
    uint32_t *early;             // [B*R] node known rejected before its parent row resolved
    unsigned long long *req_mask;   // [B] rows resolved (mask decisions, R <= 64)
    uint32_t *reset_base;
    uint32_t reset_words;
    RowStat *rowstat;            // [B*R]
    Partial *partial;            // [B*R*nsub]
    float *bmaxA;                // [B*R*nblk] block maxima (sampled rows)
    float *bsumA;                // [B*R*nblk] block sums of 2^((z - M) c2)
    float *bsumB;                // [B*nblk]   residual block sums
    unsigned long long logits_end;
    unsigned long long q_end;
    int B, R, V, D;
    int esize;
    int esub;                    // elements per A stage (24 KiB of logits)
    int nsub;                    // A stages per row
    int esb;                     // elements per B stage (24 KiB of logits + q)
    int ecb;                     // elements per B unit
    int qoff;                    // byte offset of the q area in a B stage
    int ns;                      // splits per row
    int sps;                     // A stages per split
    int ncb, nblk;
    int units_a, units_total;
    int tree;
    const int32_t *cu;           // ragged chains: request b has cu[b+1] - cu[b] drafts (null: R - 1 each)
    int total_drafts;            // ragged chains: cu[B] (packed draft rows; logit rows add one per request)
    int ahead;                   // stages the producer may have in flight
    int mask_mode;               // R <= 64: requests decide from their resolved-row mask and rows of
                                 // nodes known rejected are dropped without accounting; else every row
                                 // is streamed and a request finalises when all its rows have settled
    unsigned long long wait_ns;  // limit of every inter-block or inter-warp wait
    int16_t parent[kMaxRows];
    uint8_t depth[kMaxRows];
    uint8_t kid_off[kMaxRows + 1];   // tree: children of n are kid_list[kid_off[n] .. kid_off[n+1])
    uint8_t kid_list[kMaxRows];
};

// Stage descriptor.  The first 16 bytes are what every consumer reads per stage.
struct __align__(16) StageInfo {
    int flags;           // kind | last << 4 (last stage of its unit) | fast << 5
                         // (aligned, every element in shared memory, whole 8-element groups)
    int cnt;             // element count
    int e0;              // element offset within the row
    float c2;            // log2(e)/T, 0 for greedy
    int b, n, j;         // request, row, split (A) / chunk (B)
    int sh, tail;        // z: byte shift of element 0; elements [tail, cnt) come from global
    int shq, tailq;      // q (B)
    float m, invS;       // row statistics (B)
    int xtok;            // sampled A, last stage: token of node n+1 (-1 if none or out of range)
    float zx, qx, ux;    // ... and its logit, its draft probability, its accept uniform
    int nk;              // greedy A, first stage: children with an early-rejection check
    int ktok[kEarlyMax]; // ... their draft tokens
    int kofs[kEarlyMax]; // ... byte offset of the token's logit in its chunk at kThrOff + 16 c
                         //     (-1: token out of range, -2: not copied, read from global)
    const uint8_t *gz;
    const uint8_t *gq;
};

struct ResSlot {
    int kind, b, n, j;
    float c2;
    int xtok;
    float zx, qx, ux;
    float v[kConsumerWarps];    // greedy: lane-reduced max; sampled: warp max M_w
    int idx[kConsumerWarps];    // greedy: first index of the max
    float s[kConsumerWarps];    // sampled: warp sum of 2^((z - M_w) c2); greedy bf16: packed-record max
    int pg[kConsumerWarps];     // greedy bf16: row index of the first 8-element group holding it
};

struct Smem {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t res_full[kResSlots];
    uint64_t res_empty[kResSlots];
    StageInfo info[kStages];
    ResSlot res[kResSlots];
    uint32_t fin_rs[kEpilogueWarps][kMaxRows];   // request finalisation scratch, per epilogue warp
    int fin_tok[kEpilogueWarps][kMaxRows];
    uint8_t fin_acc[kEpilogueWarps][kMaxRows];
    int abort_flag;
    int issued;                     // stages issued by the producer
    int consumed;                   // stages released by the consumers
    int last_flag;
};

// ------------------------------------------------------- ptx wrappers --
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed(uint32_t *p, uint32_t v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_release(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t atom_add_acqrel(uint32_t *p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ unsigned long long atom_or_acqrel_u64(unsigned long long *p, unsigned long long v) {
    unsigned long long old;
    asm volatile("atom.acq_rel.gpu.global.or.b64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
    return old;
}

// 2^x by the SFU approximation (results below 2^-126 flush to zero).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void set_status(const Params &P, int bits) {
    if (P.status) atomicOr(P.status, bits);
}

// Bounded wait on an mbarrier phase; gives up (and raises the block's abort
// flag) after P.wait_ns (at the first failed try when it is 0) or as soon as
// another role has aborted.  The phase-already-complete case stays inline.
__device__ __noinline__ bool wait_bar_slow(const Params &P, Smem &S, uint64_t *bar, uint32_t parity) {
    if (P.wait_ns == 0) {
        // limit 0: one non-blocking test (try_wait may suspend the thread first)
        if (mbar_test_wait(bar, parity)) return true;
        if (!*reinterpret_cast<volatile int *>(&S.abort_flag)) {
            *reinterpret_cast<volatile int *>(&S.abort_flag) = 1;
            set_status(P, SPEC_STATUS_WAIT_TIMEOUT);
        }
        return false;
    }
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait_sleep(bar, parity, 100000u)) {
        if (*reinterpret_cast<volatile int *>(&S.abort_flag)) return false;
        if (globaltimer() - t0 > P.wait_ns) {
            *reinterpret_cast<volatile int *>(&S.abort_flag) = 1;
            set_status(P, SPEC_STATUS_WAIT_TIMEOUT);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ bool wait_bar(const Params &P, Smem &S, uint64_t *bar, uint32_t parity) {
    if (P.wait_ns != 0 && mbar_try_wait(bar, parity)) return true;
    return wait_bar_slow(P, S, bar, parity);
}

// ------------------------------------------------------------ weights --
// Per-element weights of the inverse CDF, written with explicit rounding
// intrinsics so every call site evaluates them bit-identically.  The exponent
// z*c2 - M*c2 is one fused multiply-add with nMc2 = RN(-M*c2).
// A reference max of -inf (every element -inf, e.g. a masked block) gives
// weights 2^-inf = 0 through nMc2 = 0 instead of inf - inf.
__device__ __forceinline__ float neg_mc2(float M, float c2) { return M == -INFINITY ? 0.0f : __fmul_rn(-M, c2); }

__device__ __forceinline__ float w_exp(float z, float nMc2, float c2) { return ex2(__fmaf_rn(z, c2, nMc2)); }

__device__ __forceinline__ float w_res(float z, float qv, float nmc2, float c2, float invS) {
    const float p = __fmul_rn(ex2(__fmaf_rn(z, c2, nmc2)), invS);
    return fmaxf(__fsub_rn(p, qv), 0.0f);
}

// Canonical lane partial of 8 weights: the even and the odd positions summed
// in order, then added (the order packed f32x2 accumulation produces).
__device__ __forceinline__ float lane_sum8(const float w[8]) {
    const float e = __fadd_rn(__fadd_rn(__fadd_rn(w[0], w[2]), w[4]), w[6]);
    const float o = __fadd_rn(__fadd_rn(__fadd_rn(w[1], w[3]), w[5]), w[7]);
    return __fadd_rn(e, o);
}

// Packed fp32 pairs (two IEEE operations per instruction).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t nonfinite_bf16x2(uint32_t w) {
    return __vcmpeq2(w & 0x7f807f80u, 0x7f807f80u) & ~__vcmpeq2(w, 0xff80ff80u);
}

__device__ __forceinline__ uint32_t nonfinite_f32(uint32_t w) {
    return (w & 0x7f800000u) == 0x7f800000u && w != 0xff800000u;
}

// Element view of one stage: elements [0, tail) live in shared memory at s,
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
        bad |= ((h & 0x7f80u) == 0x7f80u && h != 0xff80u);
        return __uint_as_float(static_cast<uint32_t>(h) << 16);
    } else {
        uint32_t w = (e < v.tail) ? *reinterpret_cast<const uint32_t *>(v.s + 4 * e)
                                  : __ldg(reinterpret_cast<const unsigned int *>(v.g + 4 * e));
        bad |= nonfinite_f32(w);
        return __uint_as_float(w);
    }
}

// Loads elements [e0, e0+8) of a view; returns how many are valid.
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

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

// Maxima that propagate NaN (so a NaN logit surfaces in the row max).
__device__ __forceinline__ float fmax_nan(float a, float b) {
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Max of the 8 bf16 values in a 16-byte word, by packed bf16x2 maxima.
__device__ __forceinline__ float vmax8_bf16(uint4 w) {
    uint32_t a = bmax2_nan(bmax2_nan(w.x, w.y), bmax2_nan(w.z, w.w));
    return fmax_nan(bf16_lo(a), bf16_hi(a));
}

__device__ __forceinline__ float vmax8_f32(uint4 a, uint4 b) {
    float m0 = fmax_nan(__uint_as_float(a.x), __uint_as_float(a.y));
    float m1 = fmax_nan(__uint_as_float(a.z), __uint_as_float(a.w));
    float m2 = fmax_nan(__uint_as_float(b.x), __uint_as_float(b.y));
    float m3 = fmax_nan(__uint_as_float(b.z), __uint_as_float(b.w));
    return fmax_nan(fmax_nan(m0, m1), fmax_nan(m2, m3));
}

// Warp max of a float through an order-preserving integer key and redux.
__device__ __forceinline__ int fkey(float f) {
    int b = __float_as_int(f);
    return b ^ ((b >> 31) & 0x7fffffff);
}

__device__ __forceinline__ float warp_max_redux(float v) {
    int k = __reduce_max_sync(0xffffffffu, fkey(v));
    return __int_as_float(k ^ ((k >> 31) & 0x7fffffff));
}

// (value, group) candidates: larger value wins, then the lower group.
__device__ __forceinline__ void cand_merge(float &v, int &g, float ov, int og) {
    if (ov > v || (ov == v && static_cast<unsigned>(og) < static_cast<unsigned>(g))) {
        v = ov;
        g = og;
    }
}

__device__ __forceinline__ void warp_cand(float &v, int &g) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        float ov = __shfl_xor_sync(0xffffffffu, v, off);
        int og = __shfl_xor_sync(0xffffffffu, g, off);
        cand_merge(v, g, ov, og);
    }
}

// Canonical block sum: lane partials combined by an xor butterfly; lane 0's
// value is the block's sum.
__device__ __forceinline__ float warp_butterfly_sum(float s) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, off));
    return s;
}

// Sums of N = 2 or 4 per-lane values over the warp, scattered: afterwards lane
// l holds the total of value q(l) = bits (4, 3) of l (N = 4) or bit 4 (N = 2);
// 5 dependent steps for all N values instead of 5 per value.
template <int N>
__device__ __forceinline__ float warp_sum_scatter(const float (&v)[N], int lane) {
    static_assert(N == 2 || N == 4, "2 or 4 values");
    const bool h16 = (lane & 16) != 0;
    float c;
    if constexpr (N == 4) {
        float k0 = h16 ? v[2] : v[0], k1 = h16 ? v[3] : v[1];
        const float d0 = h16 ? v[0] : v[2], d1 = h16 ? v[1] : v[3];
        k0 = __fadd_rn(k0, __shfl_xor_sync(0xffffffffu, d0, 16));
        k1 = __fadd_rn(k1, __shfl_xor_sync(0xffffffffu, d1, 16));
        const bool h8 = (lane & 8) != 0;
        c = h8 ? k1 : k0;
        const float d = h8 ? k0 : k1;
        c = __fadd_rn(c, __shfl_xor_sync(0xffffffffu, d, 8));
    } else {
        c = h16 ? v[1] : v[0];
        const float d = h16 ? v[0] : v[1];
        c = __fadd_rn(c, __shfl_xor_sync(0xffffffffu, d, 16));
        c = __fadd_rn(c, __shfl_xor_sync(0xffffffffu, c, 8));
    }
    c = __fadd_rn(c, __shfl_xor_sync(0xffffffffu, c, 4));
    c = __fadd_rn(c, __shfl_xor_sync(0xffffffffu, c, 2));
    c = __fadd_rn(c, __shfl_xor_sync(0xffffffffu, c, 1));
    return c;
}

// Mode-dependent device code: MODE 0 = chains in the padded layout, 1 = ragged
// chains (per-request draft counts from cu_num_draft_tokens), 2 = greedy trees.
// Each mode's kernel compiles only the paths it runs (smaller code, fewer
// run-time branches on the hot paths).
template <int MODE>
struct Dev {
static constexpr bool kTree = MODE == 2;
static constexpr bool kRagged = MODE == 1;

// ------------------------------------------------------------ topology --
static __device__ __forceinline__ int parent_of(const Params &P, int n) { return kTree ? P.parent[n] : n - 1; }
static __device__ __forceinline__ int depth_of(const Params &P, int n) { return kTree ? P.depth[n] : n; }

// Request b's first draft slot in the packed per-draft inputs (tokens, accept
// uniforms, q rows) and its number of drafts.  Padded batches: b * (R - 1) and
// R - 1.  Ragged chains read the offsets; offsets outside [0, total] or a count
// above R - 1 are clamped (and flagged) so no read leaves the inputs.
static __device__ __forceinline__ void draft_span(const Params &P, int b, int &first, int &count) {
    if (!kRagged) {
        first = b * (P.R - 1);
        count = P.R - 1;
        return;
    }
    int lo = __ldg(P.cu + b), hi = __ldg(P.cu + b + 1);
    const int lo0 = lo, hi0 = hi;
    lo = min(max(lo, 0), P.total_drafts);
    hi = min(max(hi, lo), P.total_drafts);
    hi = min(hi, lo + P.R - 1);
    if (lo != lo0 || hi != hi0) set_status(P, SPEC_STATUS_BAD_OFFSETS);
    first = lo;
    count = hi - lo;
}

// Rows (nodes) of request b: drafts + 1.
static __device__ __forceinline__ int rows_of(const Params &P, int b) {
    if (!kRagged) return P.R;
    int first, count;
    draft_span(P, b, first, count);
    return count + 1;
}

// Input row of node n of request b in the logits (packed: each request's rows
// follow its drafts' offsets, one extra row per request).
static __device__ __forceinline__ size_t in_row(const Params &P, int b, int n) {
    if (!kRagged) return static_cast<size_t>(b) * P.R + n;
    int first, count;
    draft_span(P, b, first, count);
    return static_cast<size_t>(first) + b + n;
}

// Per-draft input index of draft slot i (node i + 1) of request b.
static __device__ __forceinline__ size_t in_draft(const Params &P, int b, int i) {
    if (!kRagged) return static_cast<size_t>(b) * (P.R - 1) + i;
    int first, count;
    draft_span(P, b, first, count);
    return static_cast<size_t>(first) + i;
}

static __device__ __forceinline__ int node_token(const Params &P, int b, int n) {
    return __ldg(P.tokens + in_draft(P, b, n - 1));
}

// Edge parent -> child accepted, given the parent's resolved row state.
static __device__ __forceinline__ bool edge_ok(uint32_t rs, bool greedy, int child_token) {
    if (!(rs & kResolved)) return false;
    return greedy ? (static_cast<int>(rs & kIdxMask) == child_token) : ((rs & 1u) != 0u);
}

static __device__ __forceinline__ bool is_greedy(const Params &P, int b) {
    return !P.temperature || !(__ldg(P.temperature + b) > 0.0f);
}

// ---------------------------------------------------- inverse-CDF search --
// Block weights of one row: residual block sums (bmax == null), or exp block
// sums scaled by 2^((M_beta - m) c2), M_beta the block's own max.
struct BlockSource {
    const float *bsum;
    const float *bmax;
    float m, c2;
};

// 2^((M_beta - m) c2) for a block maximum M_beta (exp weights), 1 for residuals.
static __device__ __forceinline__ float block_factor_of(const BlockSource &S, float bm) {
    return S.bmax ? ex2(__fmul_rn(__fsub_rn(bm, S.m), S.c2)) : 1.0f;
}

static __device__ __forceinline__ float block_factor(const BlockSource &S, int beta) {
    return block_factor_of(S, S.bmax ? __ldcg(S.bmax + beta) : 0.0f);
}

static __device__ __forceinline__ tf block_weight(const BlockSource &S, int beta) {
    return tf_prod(__ldcg(S.bsum + beta), block_factor(S, beta));
}

static constexpr int kLocBatch = 16;   // block sums a lane loads at once (one round trip at V = 128256)

// Warp-wide: total weight and the block holding t = u * total.  Returns the
// total; beta/base receive the block and the weight before it (all lanes).
// Lane l owns blocks [l*per, (l+1)*per); the lane whose range holds t is then
// scanned by the whole warp, one block per lane.  Sums and prefixes are
// two-float.
static __device__ tf locate_block(const BlockSource &S, int nblk, float u, int lane, int &beta, tf &base) {
    const int per = (nblk + 31) / 32;
    const int lo = lane * per;
    const int hi = min(nblk, lo + per);
    // the lane's block sums and maxima are loaded kLocBatch at a time
    // (independent loads in flight together), then added in block order
    tf s = tf_of(0.0f);
    for (int i0 = lo; i0 < hi; i0 += kLocBatch) {
        float bs[kLocBatch], bm[kLocBatch];
#pragma unroll
        for (int j = 0; j < kLocBatch; ++j) {
            const int i = i0 + j;
            bs[j] = i < hi ? __ldcg(S.bsum + i) : 0.0f;
            bm[j] = (S.bmax && i < hi) ? __ldcg(S.bmax + i) : 0.0f;
        }
#pragma unroll
        for (int j = 0; j < kLocBatch; ++j)
            if (i0 + j < hi) s = tf_add(s, tf_prod(bs[j], block_factor_of(S, bm[j])));
    }
    const tf incl = warp_incl_scan_tf(s, lane);
    const tf excl = tf_add(incl, tf_neg(s));
    const tf total = tf_shfl(incl, 31);
    const tf t = tf_mulf(total, u);
    const unsigned over = __ballot_sync(0xffffffffu, tf_gt(incl, t) && hi > lo);
    const unsigned nonzero = __ballot_sync(0xffffffffu, s.h > 0.0f);
    const int L = over ? (__ffs(over) - 1) : (nonzero ? 31 - __clz(nonzero) : 0);
    const int Llo = L * per;
    const int Lhi = min(nblk, Llo + per);
    const tf Lexcl = tf_shfl(excl, L);
    int bsel = -1;
    tf bbase = Lexcl;
    int last_sel = -1;            // last block with weight seen (clamp when rounding leaves t past the end)
    tf last_base = Lexcl;
    for (int c0 = Llo; c0 < Lhi && bsel < 0; c0 += 32) {
        const int i = c0 + lane;
        const tf w = (i < Lhi) ? block_weight(S, i) : tf_of(0.0f);
        const tf wi = warp_incl_scan_tf(w, lane);
        const tf run = tf_add(bbase, tf_add(wi, tf_neg(w)));
        const unsigned cross = __ballot_sync(0xffffffffu, i < Lhi && w.h > 0.0f && tf_gt(tf_add(run, w), t));
        const unsigned pos = __ballot_sync(0xffffffffu, i < Lhi && w.h > 0.0f);
        if (cross) {
            const int q = __ffs(cross) - 1;
            bsel = c0 + q;
            bbase = tf_shfl(run, q);
        } else {
            if (pos) {
                const int q = 31 - __clz(pos);
                last_sel = c0 + q;
                last_base = tf_shfl(run, q);
            }
            bbase = tf_add(bbase, tf_shfl(wi, 31));
        }
    }
    if (bsel < 0) {
        bsel = last_sel >= 0 ? last_sel : (Llo < nblk ? Llo : 0);
        bbase = last_sel >= 0 ? last_base : Lexcl;
    }
    beta = bsel;
    base = bbase;
    return total;
}

// Warp-wide scan inside block beta of row (b, row): the first element whose
// running weight exceeds t.  residual == false: exp weights relative to the
// block max, scaled by the block factor; residual == true: max(0, p - q).
static __device__ int scan_block(const Params &P, const BlockSource &S, int b, int row, int beta, tf base, tf t,
                          bool residual, float invS, int lane) {
    const size_t rowz = in_row(P, b, row) * static_cast<size_t>(P.V);
    const int e0 = beta * kBlk + lane * 8;
    float w[8];
    const float nMc2 = neg_mc2(residual ? S.m : __ldcg(S.bmax + beta), S.c2);
    const float fac = residual ? 1.0f : block_factor(S, beta);
    const float *qrow =
        residual ? P.q + in_draft(P, b, row) * static_cast<size_t>(P.V) : nullptr;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        int e = e0 + i;
        float wi = 0.0f;
        if (e < P.V) {
            float z = logit_global(P, rowz + e);
            wi = residual ? w_res(z, __ldg(qrow + e), nMc2, S.c2, invS) : w_exp(z, nMc2, S.c2);
        }
        w[i] = wi;
    }
    const float s = lane_sum8(w);
    const tf ls = tf_prod(s, fac);
    const tf incl = warp_incl_scan_tf(ls, lane);
    const tf lbase = tf_add(base, tf_add(incl, tf_neg(ls)));
    unsigned hit = __ballot_sync(0xffffffffu, tf_gt(tf_add(lbase, ls), t) && s > 0.0f);
    unsigned pos = __ballot_sync(0xffffffffu, s > 0.0f);
    int L = hit ? (__ffs(hit) - 1) : (pos ? 31 - __clz(pos) : 0);
    int j = -1;
    if (lane == L) {
        tf acc = lbase;
        int last_pos = 0;
        for (int i = 0; i < 8; ++i) {
            if (w[i] > 0.0f) last_pos = i;
            acc = tf_add(acc, tf_prod(w[i], fac));
            if (hit && w[i] > 0.0f && tf_gt(acc, t)) {
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

// Sample one token from row `row` of request b (warp-wide): residual weights
// if `residual` (falling back to p when the residual has no mass), else p.
static __device__ int sample_row(const Params &P, int b, int row, bool residual, float u, int lane) {
    const size_t ri = static_cast<size_t>(b) * P.R + row;
    const float m = __ldcg(&P.rowstat[ri].m);
    const float Sh = __ldcg(&P.rowstat[ri].Sh);
    const float c2 = kLog2e / __ldg(P.temperature + b);
    int beta;
    tf base;
    if (residual) {
        BlockSource S{P.bsumB + static_cast<size_t>(b) * P.nblk, nullptr, m, c2};
        const tf Z = locate_block(S, P.nblk, u, lane, beta, base);
        if (Z.h > 0.0f) return scan_block(P, S, b, row, beta, base, tf_mulf(Z, u), true, 1.0f / Sh, lane);
    }
    BlockSource S{P.bsumA + ri * P.nblk, P.bmaxA + ri * P.nblk, m, c2};
    const tf tot = locate_block(S, P.nblk, u, lane, beta, base);
    return scan_block(P, S, b, row, beta, base, tf_mulf(tot, u), false, 0.0f, lane);
}

// --------------------------------------------------- request finalisation --
// Warp-wide: row states and node tokens of request b into the warp's scratch
// (after the caller's acquire of every row it will use).  Returns whether a
// draft token is outside [0, V).
static __device__ bool load_request(const Params &P, Smem &S, int slot, int b, int Rb, int lane) {
    uint32_t *rs = S.fin_rs[slot];
    int *tok = S.fin_tok[slot];
    int range_bad = 0;
    for (int i = lane; i < Rb; i += 32) {
        rs[i] = ld_acquire(P.rowstate + static_cast<size_t>(b) * P.R + i);
        tok[i] = i > 0 ? node_token(P, b, i) : -1;
        if (i > 0 && (tok[i] < 0 || tok[i] >= P.V)) range_bad = 1;
    }
    __syncwarp();
    return __any_sync(0xffffffffu, range_bad) != 0;
}

// Warp-wide.  Request b is decided (every row its outcome depends on is
// resolved): walk the tree, write the outputs, publish the decision (and draw
// the bonus token of a sampled request that accepted every draft).  With
// `loaded`, the warp's scratch already holds the request's states and tokens
// and range_bad says whether a token was out of range.
template <bool SMP>
static __device__ int finalize_request(const Params &P, Smem &S, int slot, int b, int lane, bool loaded,
                                             bool range_bad) {
    uint32_t *rs = S.fin_rs[slot];
    int *tok = S.fin_tok[slot];
    uint8_t *acc = S.fin_acc[slot];
    const int Rb = rows_of(P, b);
    if (!loaded) range_bad = load_request(P, S, slot, b, Rb, lane);
    if (range_bad && lane == 0) set_status(P, SPEC_STATUS_TOKEN_RANGE);
    __syncwarp();
    const bool greedy = !SMP || is_greedy(P, b);
    int bonus = 0;
    uint32_t decision = kDecided;
    if (lane == 0) {
        acc[0] = 1;
        int best = 0;
        for (int i = 1; i < Rb; ++i) {
            int p = parent_of(P, i);
            bool ok = acc[p] && edge_ok(rs[p], greedy, tok[i]);
            acc[i] = ok;
            if (ok && depth_of(P, i) > depth_of(P, best)) best = i;
        }
        const int d = depth_of(P, best);
        int32_t *ot = P.out_tokens + static_cast<size_t>(b) * (P.D + 1);
        int32_t *op = P.out_path ? P.out_path + static_cast<size_t>(b) * (P.D + 1) : nullptr;
        int node = best;
        for (int i = d; i >= 1; --i) {
            ot[i - 1] = tok[node];
            if (op) op[i] = node;
            node = parent_of(P, node);
        }
        if (op) {
            op[0] = 0;
            for (int i = d + 1; i <= P.D; ++i) op[i] = -1;
        }
        for (int i = d + 1; i <= P.D; ++i) ot[i] = -1;
        if (greedy) {
            uint32_t r = rs[best];
            ot[d] = (r & kResolved) ? static_cast<int>(r & kIdxMask) : 0;
        } else if (d < Rb - 1) {
            // ot[d] is the residual pass's (which may already have run: the decision
            // can be published as soon as the rejecting row resolves)
            decision |= kNeedsResidual | static_cast<uint32_t>(d);
        } else {
            bonus = 1;
        }
        P.out_count[b] = kTree ? d + 1 : d;
        acc[0] = static_cast<uint8_t>(d < 255 ? d : 255);   // accepted count for the slot fix-up below
    }
    bonus = __shfl_sync(0xffffffffu, bonus, 0);
    if (P.slots && !kTree) {
        // the slot_mapping fix-up fused here: request b's slots 0..a keep their
        // values (row 0 is the last accepted token), the rest become padding
        __syncwarp();
        const int a = acc[0];
        int64_t *sl = P.slots + in_row(P, b, 0);
        for (int j = a + 1 + lane; j < Rb; j += 32) sl[j] = P.pad;
    }
    if (lane == 0) {
        // Residual units read the decision and then this request's row data:
        // publish with release.  Without residual units nobody waits on it.
        if (P.units_total > P.units_a) st_release(P.req_state + b, decision);
        else st_relaxed(P.req_state + b, decision);
    }
    __syncwarp();
    // a sampled request that accepted every draft draws its bonus token from the
    // last row; the caller draws it (one draw site per kernel)
    return (SMP && bonus) ? Rb - 1 : -1;
}

// Counting decisions (R > 64): one more row of request b has settled; true
// when it was the request's last (every row resolved: the request is decided).
static __device__ __forceinline__ bool settle_row(const Params &P, int b, int lane) {
    uint32_t old = 0;
    if (lane == 0) old = atom_add_acqrel(P.req_ctr + b, 1u);
    old = __shfl_sync(0xffffffffu, old, 0);
    return old == static_cast<uint32_t>(rows_of(P, b) - 1);
}

// Chains: with the rows of mask m resolved (rows 0..r-1, r its trailing ones),
// is request b decided?  Yes once one of rows 0..r-1 rejects its draft
// (notacc: rows whose draft is not accepted), or every row is resolved.
static __device__ __forceinline__ bool chain_decided(unsigned long long m, int Rb, unsigned long long notacc) {
    const int r = (~m == 0ull) ? 64 : __ffsll(static_cast<long long>(~m)) - 1;
    const int f = notacc ? __ffsll(static_cast<long long>(notacc)) - 1 : 64;
    return f < r || r >= Rb;
}

// Greedy trees: with the rows of mask m resolved, is the request decided?
// Yes once every accepted node (the root; a child whose parent is accepted and
// resolved with an argmax equal to the child's token) is resolved.  Warp-wide:
// lane l holds nodes l and l + 32; the accepted set grows one level per step.
static __device__ __forceinline__ bool tree_decided(const Params &P, const uint32_t *rs, const int *tok, int Rb,
                                                    unsigned long long m, int lane) {
    bool e[2];
    int par[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int c = lane + 32 * h;
        par[h] = (c >= 1 && c < Rb) ? P.parent[c] : 0;
        e[h] = c >= 1 && c < Rb && ((m >> par[h]) & 1ull) && edge_ok(rs[par[h]], true, tok[c]);
    }
    unsigned long long a = 1ull;
    for (int step = 0; step < 64; ++step) {
        const unsigned long long na =
            1ull | static_cast<unsigned long long>(__ballot_sync(0xffffffffu, e[0] && ((a >> par[0]) & 1ull))) |
            (static_cast<unsigned long long>(__ballot_sync(0xffffffffu, e[1] && ((a >> par[1]) & 1ull))) << 32);
        if (na == a) break;
        a = na;
    }
    return (a & ~m) == 0ull;
}

// Mask decisions (R <= 64): row n of request b is resolved (its state written by
// this warp's lane 0).  One atomic adds it to the request's mask; true for the
// warp whose row turns the request from undecided to decided (it finalises the
// request; the request's states and tokens are then in its scratch, and
// range_bad says whether a token was out of range).  Rows of nodes known
// rejected are never streamed and never recorded: nothing waits for them.
static __device__ bool record_row(const Params &P, Smem &S, int slot, int b, int n, bool greedy, int lane,
                           bool &range_bad) {
    unsigned long long old = 0;
    if (lane == 0) old = atom_or_acqrel_u64(P.req_mask + b, 1ull << n);
    old = (static_cast<unsigned long long>(__shfl_sync(0xffffffffu, static_cast<uint32_t>(old >> 32), 0)) << 32) |
          __shfl_sync(0xffffffffu, static_cast<uint32_t>(old), 0);
    const unsigned long long now = old | (1ull << n);
    // Only a row that can change the outcome needs the request's states: for a
    // chain the row that extends the resolved prefix, for a tree a row whose
    // parent is resolved (or the root).
    if (kTree) {
        if (n > 0 && !((old >> P.parent[n]) & 1ull)) return false;
    } else {
        const int r_old = (~old == 0ull) ? 64 : __ffsll(static_cast<long long>(~old)) - 1;
        if (n != r_old) return false;
    }
    __syncwarp();   // the whole warp reads after lane 0's acquire
    const int Rb = rows_of(P, b);
    range_bad = load_request(P, S, slot, b, Rb, lane);
    const uint32_t *rs = S.fin_rs[slot];
    const int *tok = S.fin_tok[slot];
    bool turn;
    if (kTree) {
        turn = tree_decided(P, rs, tok, Rb, now, lane) && !tree_decided(P, rs, tok, Rb, old, lane);
    } else {
        unsigned long long notacc = 0;
        for (int base = 0; base < Rb - 1; base += 32) {
            const int i = base + lane;
            const bool na = i < Rb - 1 && !edge_ok(rs[i], greedy, tok[i + 1]);
            notacc |= static_cast<unsigned long long>(__ballot_sync(0xffffffffu, na)) << base;
        }
        turn = chain_decided(now, Rb, notacc) && !chain_decided(old, Rb, notacc);
    }
    return turn;
}

// A row is done: record it (mask decisions) or settle it (counting), and
// finalise the request if this row decided it.  Returns the row of a bonus draw
// the caller must make, or -1.
template <bool SMP>
static __device__ __forceinline__ int finish_row(const Params &P, Smem &S, int slot, int b, int n, bool greedy, int lane) {
    bool range_bad = false;
    const bool loaded = P.mask_mode != 0;
    const bool fin = loaded ? record_row(P, S, slot, b, n, greedy, lane, range_bad) : settle_row(P, b, lane);
    return fin ? finalize_request<SMP>(P, S, slot, b, lane, loaded, range_bad) : -1;
}

// Warp-wide: resolve row n of request b once all its splits are in.
// Greedy: gidx is the row's argmax (first index), gmax its value.  Sampled:
// (m, Srow) are the row statistics and (xtok, zx, qx, ux) the operands of the
// accept test of node n+1 (xtok < 0: no child, or its token is out of range).
template <bool SMP>
static __device__ void resolve_row(const Params &P, int b, int n, bool greedy, float c2, int gidx, float gmax, float m,
                            tf Srow, int xtok, float zx, float qx, float ux, int lane) {
    const size_t ri = static_cast<size_t>(b) * P.R + n;
    const int Rb = rows_of(P, b);
    if (lane == 0) {
        uint32_t rsv;
        if (!SMP || greedy) {
            const int g = (gidx < 0 || gidx >= P.V) ? 0 : gidx;
            rsv = kResolved | static_cast<uint32_t>(g);
            if (!isfinite(gmax)) set_status(P, SPEC_STATUS_NONFINITE);
        } else {
            if (!isfinite(m) || !isfinite(Srow.h)) set_status(P, SPEC_STATUS_NONFINITE);
            RowStat st;
            st.m = m;
            st.Sh = Srow.h;
            st.Sl = Srow.l;
            st.pad = 0.0f;
            P.rowstat[ri] = st;
            uint32_t acc = 0;
            if (n < Rb - 1) {
                if (xtok < 0) {
                    set_status(P, SPEC_STATUS_TOKEN_RANGE);
                } else if (qx == 0.0f) {
                    acc = 1;
                } else {
                    // u < p(x) / q(x) with p(x) = e(x) / S, multiplied through by q(x) S > 0
                    const float ex = ex2(__fmul_rn(__fsub_rn(zx, m), c2));
                    acc = ux * (qx * Srow.h) < ex;
                }
            }
            rsv = kResolved | acc;
        }
        // Relaxed: skip checks use only the value; readers of the row's data (block
        // sums and maxima, statistics) synchronise through the atomic that follows
        // (the mask OR or the settle add: acq_rel, same thread, cumulative over the
        // consumers' writes this warp observed at the stage barrier) or through a
        // decision this thread publishes with release.
        st_relaxed(P.rowstate + ri, rsv);
    }
    __syncwarp();
}

// --------------------------------------------------------------- roles --
// Producer (warp 0).  What the producer needs of an A unit before streaming it,
// loaded one stage ahead so the loads are in flight while the previous unit's
// last stage streams: lane i (and i + 32) holds edge i of the unit's path
// counted from the node upwards (the early-rejection flag of the edge's child,
// the state of its parent row, the child's token); lane c < kEarlyMax the token
// of child c (greedy rows: the consumers' early-rejection check); every lane the
// request's temperature; lane 0, for a sampled row, node n+1's token and accept
// uniform.
struct Ahead {
    int u;                       // unit, or -1 when none is known
    int b, n, j;                 // request, node, split (A units)
    int check;                   // the node's path is checked before it is streamed
    int echild[2];
    uint32_t ef[2], rs[2];
    int etok[2];
    int ktok;
    float temp;
    int xtok;
    float ux;
};

static __device__ void ahead_load(const Params &P, Ahead &A, int u, bool check, int lane) {
    A.u = u;
    A.check = 0;
    A.ktok = -1;
    A.temp = 0.0f;
    A.xtok = -1;
    A.ux = 0.0f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        A.ef[h] = 0u;
        A.rs[h] = 0u;
        A.etok[h] = -1;
        A.echild[h] = 0;
    }
    if (u < 0 || u >= P.units_a) return;
    const int per_node = P.B * P.ns;
    const int n = u / per_node;
    const int rem = u - n * per_node;
    const int b = rem / P.ns;
    A.n = n;
    A.b = b;
    A.j = rem - b * P.ns;
    int first, count;   // request b's drafts: tokens[first + i] is node i + 1's token
    draft_span(P, b, first, count);
    const int Rb = count + 1;
    if (n >= Rb) return;   // ragged: this request has fewer rows
    if (P.temperature) A.temp = __ldg(P.temperature + b);
    // children's tokens (greedy early-rejection check)
    int nk, k0 = 0;
    if (kTree) {
        k0 = P.kid_off[n];
        nk = P.kid_off[n + 1] - k0;
    } else {
        nk = n < Rb - 1 ? 1 : 0;
    }
    if (lane < min(nk, kEarlyMax))
        A.ktok = __ldg(P.tokens + first + (kTree ? static_cast<int>(P.kid_list[k0 + lane]) : n + 1) - 1);
    if (P.u_accept && lane == 0 && n < Rb - 1) {
        A.xtok = __ldg(P.tokens + first + n);
        A.ux = __ldg(P.u_accept + first + n);
    }
    if (!check || n == 0) return;
    A.check = 1;
    const int d = depth_of(P, n);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int i = lane + 32 * h;
        if (i < d) {
            int child = n;
            if (kTree) {
#pragma unroll 1
                for (int q = 0; q < i; ++q) child = P.parent[child];
            } else {
                child = n - i;
            }
            A.echild[h] = child;
            A.etok[h] = __ldg(P.tokens + first + child - 1);
        }
    }
}

// The changing facts of the unit's path (early-rejection flags, parent row
// states): loaded when the unit is about to start, so they are as fresh as
// possible; they arrive while the producer waits for the unit's first slot.
static __device__ __forceinline__ void check_issue(const Params &P, Ahead &A, int lane) {
    if (!A.check) return;
    const size_t rb = static_cast<size_t>(A.b) * P.R;
    const int d = depth_of(P, A.n);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        if (lane + 32 * h < d) {
            A.ef[h] = ld_relaxed(P.early + rb + A.echild[h]);
            A.rs[h] = ld_relaxed(P.rowstate + rb + parent_of(P, A.echild[h]));
        }
    }
}

// Is the A unit's node known to be rejected?  (An edge on its path flagged
// early, or rejected by its resolved parent row.)  Warp-wide.
static __device__ __forceinline__ bool ahead_dead(const Ahead &A, bool greedy) {
    bool bad = false;
#pragma unroll
    for (int h = 0; h < 2; ++h)
        bad |= A.ef[h] != 0u || ((A.rs[h] & kResolved) && !edge_ok(A.rs[h], greedy, A.etok[h]));
    return A.check && __any_sync(0xffffffffu, bad);
}

// Copy geometry: 16-byte aligned bulk range covering [g, g + cnt*es), clipped
// to the tensor's last full 16 bytes; elements past the clip come from global.
static __device__ __forceinline__ void copy_geom(const uint8_t *g, int cnt, int es, unsigned long long end, int &sh,
                                          int &tail, const uint8_t *&src, uint32_t &nbytes) {
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
}

template <int ES, bool SMP>
static __device__ void producer(const Params &P, Smem &S, uint8_t *ring, int lane) {
    int it = 0;   // stages issued
    const int claim_base = static_cast<int>(gridDim.x);
    bool aborted = false;
    unsigned long long loaded_bytes = 0;
    int a_loaded = 0, a_skipped = 0, b_loaded = 0, b_skipped = 0;
    const bool dropping = P.mask_mode != 0;   // rows of nodes known rejected are not streamed

    // Reserve the next stage: at most P.ahead stages are issued and not yet
    // released (stage it - ahead released; consumers release in order, so its
    // slot's previous use, stage it - kStages, is free too).
    auto acquire_stage = [&](int &st) -> bool {
        st = it % kStages;
        if (it >= P.ahead) {
            const int r = it - P.ahead;
            if (!wait_bar(P, S, &S.empty[r % kStages], static_cast<uint32_t>((r / kStages) & 1))) return false;
        }
        return true;
    };

    // Claims run ahead of the work: the claim for the unit after `cur` is issued
    // one stage before that unit's lookahead loads, which go out with cur's last
    // stage (so with one-stage units, the claim goes out with the previous
    // unit's stage).  A block holds at most two claimed units it has not started.
    int pc = 0;               // lane 0: result of the claim in flight
    bool pc_live = false;     // a claim is in flight
    auto claim_issue = [&]() {
        if (lane == 0) pc = claim_base + static_cast<int>(atomicAdd(P.ctrl + 0, 1u));
        pc_live = true;
    };
    Ahead cur, nxt;
    bool nxt_known = false;
    bool checks = false;      // the block's first unit is not checked: nothing can be known yet
    // The next unit: take its claim (issuing it if none is in flight) and load its
    // lookahead facts; with one-stage units, claim the unit after it at once.
    auto advance_next = [&](bool one_stage) {
        if (nxt_known) return;
        if (!pc_live) claim_issue();
        const int v = __shfl_sync(0xffffffffu, pc, 0);
        pc_live = false;
        ahead_load(P, nxt, v, dropping && checks, lane);
        checks = true;
        nxt_known = true;
        if (one_stage && v < P.units_total) claim_issue();
    };
    // The first unit is static (block b takes unit b) and is never dropped: before
    // anything else, its first stages start moving into L2, so HBM is busy while
    // the producer sets up (its bulk copies then find the bytes on chip).
    if (lane == 0 && !kRagged && static_cast<int>(blockIdx.x) < P.units_a) {
        const int u0 = static_cast<int>(blockIdx.x);
        const int n0 = u0 / (P.B * P.ns);
        const int r0 = u0 - n0 * (P.B * P.ns);
        const int b0 = r0 / P.ns;
        const int s0 = (r0 - b0 * P.ns) * P.sps;
        const int ns0 = min(min(P.nsub, s0 + P.sps) - s0, P.ahead);
        const int e0 = s0 * P.esub;
        const int e1 = min(P.V, e0 + ns0 * P.esub);
        const unsigned long long a0 =
            reinterpret_cast<unsigned long long>(P.logits) + (in_row(P, b0, n0) * P.V + e0) * ES;
        const unsigned long long lo = a0 & ~15ull;
        const unsigned long long hi = min((a0 + static_cast<unsigned long long>(e1 - e0) * ES + 15ull) & ~15ull,
                                          P.logits_end & ~15ull);
        if (hi > lo) bulk_prefetch_l2(reinterpret_cast<const void *>(lo), static_cast<uint32_t>(hi - lo));
    }
    // the next unit is claimed at once
    pc = static_cast<int>(blockIdx.x);
    pc_live = true;
    advance_next(true);
    cur = nxt;
    nxt_known = false;

    while (!aborted) {
        const int u = cur.u;
        if (u < 0 || u >= P.units_total) break;
        if (u < P.units_a) {
            // ---------------- A unit: split j of row n of request b
            const int n = cur.n, b = cur.b, j = cur.j;
            const int s0 = j * P.sps;
            const int s1 = min(P.nsub, s0 + P.sps);
            const bool one_stage = P.sps == 1;
            bool skip = kRagged && n >= rows_of(P, b);   // ragged: this request has fewer rows
            const bool greedy = !SMP || !(cur.temp > 0.0f);
            const float c2 = greedy ? 0.0f : kLog2e / cur.temp;
            int st0 = -1;   // the first stage's slot, reserved while the check's loads fly
            if (!skip && dropping) {
                check_issue(P, cur, lane);
                if (!acquire_stage(st0)) {
                    aborted = true;
                    break;
                }
                if (ahead_dead(cur, greedy)) {
                    skip = true;
                    ++a_skipped;
                }
            }
            if (skip) {
                advance_next(one_stage);
                cur = nxt;
                nxt_known = false;
                continue;
            }
            ++a_loaded;
            const size_t rowe = in_row(P, b, n) * static_cast<size_t>(P.V);
            // accept-test operands of node n+1 (sampled rows): loaded now, written
            // into the unit's last stage (the loads overlap the stage waits)
            float zx = 0.0f, qx = 0.0f;
            const int xtok = (!greedy && cur.xtok >= 0 && cur.xtok < P.V) ? cur.xtok : -1;
            if (SMP && lane == 0 && !greedy && xtok >= 0) {
                zx = logit_global(P, rowe + static_cast<size_t>(xtok));
                qx = __ldg(P.q + in_draft(P, b, n) * P.V + static_cast<size_t>(xtok));
            }
            int nk = 0;
            if (greedy) {
                if (kTree) nk = P.kid_off[n + 1] - P.kid_off[n];
                else nk = n < rows_of(P, b) - 1 ? 1 : 0;
                nk = min(nk, kEarlyMax);
            }
            for (int s = s0; s < s1; ++s) {
                int st = st0;
                if (s != s0 || st0 < 0) {
                    if (!acquire_stage(st)) {
                        aborted = true;
                        break;
                    }
                }
                const bool last = (s == s1 - 1);
                if (s == max(s0, s1 - 2) && !one_stage && !last && !pc_live && !nxt_known) claim_issue();
                if (lane == 0) {
                    StageInfo &I = S.info[st];
                    I.b = b;
                    I.n = n;
                    I.j = j;
                    I.e0 = s * P.esub;
                    I.cnt = min(P.esub, P.V - I.e0);
                    I.c2 = c2;
                    I.xtok = xtok;
                    if (last) {
                        I.zx = zx;
                        I.qx = qx;
                        I.ux = cur.ux;
                    }
                    I.gz = P.logits + (rowe + I.e0) * ES;
                    const uint8_t *src;
                    uint32_t nb;
                    copy_geom(I.gz, I.cnt, ES, P.logits_end, I.sh, I.tail, src, nb);
                    const int fast = (I.sh == 0 && I.tail == I.cnt && (I.cnt & 7) == 0);
                    I.flags = kA | (static_cast<int>(last) << 4) | (fast << 5) | (s == s0 ? kFirstF : 0u);
                    loaded_bytes += nb;
                    fence_proxy_async();
                    uint8_t *dst = ring + static_cast<size_t>(st) * kStageBytes;
                    if (s != s0) {
                        if (nb) {
                            mbar_expect_tx(&S.full[st], nb);
                            bulk_g2s(dst, src, nb, &S.full[st]);
                        } else {
                            mbar_arrive(&S.full[st]);
                        }
                    } else if (nb) {
                        // first stage: the row's copy goes out at once; the stage
                        // completes only after the arrive below
                        mbar_expect_tx_only(&S.full[st], nb);
                        bulk_g2s(dst, src, nb, &S.full[st]);
                    }
                }
                if (s == s0) {
                    // the children's logits travel with the first stage
                    int kt[kEarlyMax];
#pragma unroll
                    for (int c = 0; c < kEarlyMax; ++c) kt[c] = __shfl_sync(0xffffffffu, cur.ktok, c);
                    if (lane == 0) {
                        StageInfo &I = S.info[st];
                        uint8_t *dst = ring + static_cast<size_t>(st) * kStageBytes;
                        uint32_t extra = 0;
                        const uint8_t *ksrc[kEarlyMax];
                        I.nk = nk;
#pragma unroll
                        for (int c = 0; c < kEarlyMax; ++c) {
                            I.ktok[c] = kt[c];
                            int ko = -1;
                            ksrc[c] = nullptr;
                            if (c < nk && kt[c] >= 0 && kt[c] < P.V) {
                                const unsigned long long a = reinterpret_cast<unsigned long long>(P.logits) +
                                                             (rowe + static_cast<size_t>(kt[c])) * ES;
                                const unsigned long long ch = a & ~15ull;
                                if (ch + 16 <= P.logits_end) {
                                    ko = static_cast<int>(a - ch);
                                    ksrc[c] = reinterpret_cast<const uint8_t *>(ch);
                                    extra += 16;
                                } else {
                                    ko = -2;
                                }
                            }
                            I.kofs[c] = ko;
                        }
                        if (extra) {
                            mbar_expect_tx(&S.full[st], extra);
#pragma unroll
                            for (int c = 0; c < kEarlyMax; ++c)
                                if (ksrc[c]) bulk_g2s(dst + kThrOff + 16 * c, ksrc[c], 16, &S.full[st]);
                        } else {
                            mbar_arrive(&S.full[st]);
                        }
                    }
                }
                ++it;
                if (last) advance_next(one_stage);   // the next unit's lookahead rides on this stage
            }
            if (aborted) break;
        } else if (SMP) {
            // ---------------- B unit: chunk c of the rejected row of request b
            const int v = u - P.units_a;
            const int b = v / P.ncb;
            const int c = v - b * P.ncb;
            uint32_t stv = 0;
            if (lane == 0) {
                stv = ld_acquire(P.req_state + b);
                if (!(stv & kDecided)) {
                    unsigned long long t0 = globaltimer();
                    while (!(stv & kDecided)) {
                        if (P.wait_ns == 0 || globaltimer() - t0 > P.wait_ns) break;
                        __nanosleep(200);
                        stv = ld_acquire(P.req_state + b);
                    }
                    if (!(stv & kDecided)) set_status(P, SPEC_STATUS_WAIT_TIMEOUT);
                }
            }
            stv = __shfl_sync(0xffffffffu, stv, 0);
            const int a = static_cast<int>(stv & kIdxMask);
            if (!(stv & kDecided) || !(stv & kNeedsResidual) || a >= rows_of(P, b) - 1) {
                ++b_skipped;
                advance_next(false);
            } else {
                ++b_loaded;
                const size_t ri = static_cast<size_t>(b) * P.R + a;
                const float m = __ldcg(&P.rowstat[ri].m);
                const float Sh = __ldcg(&P.rowstat[ri].Sh);
                const float c2 = kLog2e / __ldg(P.temperature + b);
                const size_t rowe = in_row(P, b, a) * static_cast<size_t>(P.V);
                const size_t qrowe = in_draft(P, b, a) * static_cast<size_t>(P.V);
                const int e_begin = c * P.ecb;
                const int e_end = min(P.V, e_begin + P.ecb);
                for (int e = e_begin; e < e_end; e += P.esb) {
                    int st;
                    if (!acquire_stage(st)) {
                        aborted = true;
                        break;
                    }
                    const int last = (e + P.esb >= e_end);
                    if (!last && e + 2 * P.esb >= e_end && !pc_live && !nxt_known) claim_issue();
                    if (lane == 0) {
                        StageInfo &I = S.info[st];
                        I.b = b;
                        I.n = a;
                        I.j = c;
                        I.e0 = e;
                        I.cnt = min(P.esb, P.V - e);
                        I.c2 = c2;
                        I.m = m;
                        I.invS = 1.0f / Sh;
                        I.gz = P.logits + (rowe + e) * ES;
                        I.gq = reinterpret_cast<const uint8_t *>(P.q + qrowe + e);
                        const uint8_t *sz, *sq;
                        uint32_t nz, nq;
                        copy_geom(I.gz, I.cnt, ES, P.logits_end, I.sh, I.tail, sz, nz);
                        copy_geom(I.gq, I.cnt, 4, P.q_end, I.shq, I.tailq, sq, nq);
                        const int fast =
                            (I.sh == 0 && I.tail == I.cnt && I.shq == 0 && I.tailq == I.cnt && (I.cnt & 7) == 0);
                        I.flags = kB | (last << 4) | (fast << 5);
                        loaded_bytes += nz + nq;
                        fence_proxy_async();
                        uint8_t *dst = ring + static_cast<size_t>(st) * kStageBytes;
                        if (nz + nq) {
                            mbar_expect_tx(&S.full[st], nz + nq);
                            if (nz) bulk_g2s(dst, sz, nz, &S.full[st]);
                            if (nq) bulk_g2s(dst + P.qoff, sq, nq, &S.full[st]);
                        } else {
                            mbar_arrive(&S.full[st]);
                        }
                    }
                    ++it;
                    if (last) advance_next(false);
                }
                if (aborted) break;
            }
        } else {
            advance_next(false);
        }
        cur = nxt;
        nxt_known = false;
    }
    // End marker (not after an abort: the consumers are leaving already).
    if (!aborted) {
        int st;
        if (acquire_stage(st)) {
            if (lane == 0) {
                S.info[st].flags = kEnd;
                mbar_arrive(&S.full[st]);
            }
            ++it;
        }
    }
    if (lane == 0) {
        S.issued = it;
        if (a_loaded) atomicAdd(P.stats + 0, static_cast<unsigned long long>(a_loaded));
        if (a_skipped) atomicAdd(P.stats + 1, static_cast<unsigned long long>(a_skipped));
        if (b_loaded) atomicAdd(P.stats + 2, static_cast<unsigned long long>(b_loaded));
        if (b_skipped) atomicAdd(P.stats + 3, static_cast<unsigned long long>(b_skipped));
        if (loaded_bytes) atomicAdd(P.stats + 4, loaded_bytes);
    }
}

// Fold a finished sum s (relative to reference max M) into a warp's running
// (Mw, Sw + Sc) statistics, with Neumaier compensation.
static __device__ __forceinline__ void fold_stats(float M, float s, float c2, float &Mw, float &Sw, float &Sc) {
    if (M == -INFINITY) return;   // an all -inf stretch adds nothing
    float add;
    if (M > Mw) {
        const float f = ex2(__fmul_rn(__fsub_rn(Mw, M), c2));
        Sw = __fmul_rn(Sw, f);
        Sc = __fmul_rn(Sc, f);
        Mw = M;
        add = s;
    } else {
        add = __fmul_rn(s, ex2(__fmul_rn(__fsub_rn(M, Mw), c2)));
    }
    const float tsum = __fadd_rn(Sw, add);
    if (fabsf(Sw) >= fabsf(add)) Sc = __fadd_rn(Sc, __fadd_rn(__fsub_rn(Sw, tsum), add));
    else Sc = __fadd_rn(Sc, __fadd_rn(__fsub_rn(add, tsum), Sw));
    Sw = tsum;
}

// Does either bf16 half of a exceed the matching half of b?  (NaN: no.)
static __device__ __forceinline__ bool bf16x2_any_gt(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("{\n\t.reg .pred p, q;\n\t"
        "setp.gt.bf16x2 p|q, %1, %2;\n\t"
        "or.pred p, p, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(a), "r"(b));
    return r != 0;
}

// Packed running maximum of the two bf16 halves with the row index of the
// group that first set each half's record (branch-free): the half of `a`
// that beats the record moves it to group start ge.  NaN freezes both.
static __device__ __forceinline__ void bf16x2_record(uint32_t a, uint32_t &pk, int ge, int &glo, int &ghi) {
    asm("{\n\t.reg .pred plo, phi;\n\t"
        "setp.gt.bf16x2 plo|phi, %3, %2;\n\t"
        "selp.s32 %0, %4, %0, plo;\n\t"
        "selp.s32 %1, %4, %1, phi;\n\t}"
        : "+r"(glo), "+r"(ghi)
        : "r"(pk), "r"(a), "r"(ge));
    pk = bmax2_nan(pk, a);
}

// A bf16 value (given as its exact float) in both halves of a word.
static __device__ __forceinline__ uint32_t bf16_pair(float m) {
    const uint32_t h = __float_as_uint(m) >> 16;
    return h | (h << 16);
}

// Eight logits of a 16-byte (bf16) or 32-byte (fp32) register pair as floats.
template <int ES>
static __device__ __forceinline__ void unpack8(const uint4 a, const uint4 c, float x[8]) {
    if (ES == 2) {
        x[0] = bf16_lo(a.x); x[1] = bf16_hi(a.x);
        x[2] = bf16_lo(a.y); x[3] = bf16_hi(a.y);
        x[4] = bf16_lo(a.z); x[5] = bf16_hi(a.z);
        x[6] = bf16_lo(a.w); x[7] = bf16_hi(a.w);
    } else {
        x[0] = __uint_as_float(a.x); x[1] = __uint_as_float(a.y);
        x[2] = __uint_as_float(a.z); x[3] = __uint_as_float(a.w);
        x[4] = __uint_as_float(c.x); x[5] = __uint_as_float(c.y);
        x[6] = __uint_as_float(c.z); x[7] = __uint_as_float(c.w);
    }
}

// Greedy step over one 8-element group already in registers (row index of its
// first element: e_first).
template <int ES>
static __device__ __forceinline__ void greedy_regs(const uint4 a, const uint4 c, int e_first, float &best, int &bidx,
                                            float &mx) {
    const float m = (ES == 2) ? vmax8_bf16(a) : vmax8_f32(a, c);
    mx = fmax_nan(mx, m);
    if (m > best) {
        best = m;
        float x[8];
        unpack8<ES>(a, c, x);
        int i = 7;
#pragma unroll
        for (int q = 7; q >= 0; --q)
            if (x[q] == m) i = q;
        bidx = e_first + i;
    }
}

// Greedy step over one 8-element group: NaN-propagating max into mx, and if
// the group's max beats `best`, the group's first element equal to it.
template <int ES>
static __device__ __forceinline__ void group_step(const View &v, int g, int e_row0, bool fast, float &best, int &bidx,
                                           float &mx, uint32_t &bad) {
    if (fast) {
        if (ES == 2) {
            const uint4 w = *reinterpret_cast<const uint4 *>(v.s + 16 * g);
            const float m = vmax8_bf16(w);
            mx = fmax_nan(mx, m);
            if (m > best) {
                best = m;
                const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
                int i = 7;
#pragma unroll
                for (int q = 3; q >= 0; --q) {
                    if (bf16_hi(ww[q]) == m) i = 2 * q + 1;
                    if (bf16_lo(ww[q]) == m) i = 2 * q;
                }
                bidx = e_row0 + 8 * g + i;
            }
        } else {
            const uint4 *p = reinterpret_cast<const uint4 *>(v.s + 32 * g);
            const uint4 a = p[0], c = p[1];
            const float m = vmax8_f32(a, c);
            mx = fmax_nan(mx, m);
            if (m > best) {
                best = m;
                const uint32_t ww[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
                int i = 7;
#pragma unroll
                for (int q = 7; q >= 0; --q)
                    if (__uint_as_float(ww[q]) == m) i = q;
                bidx = e_row0 + 8 * g + i;
            }
        }
        return;
    }
    const int e0 = 8 * g;
    const int nv = min(8, v.cnt - e0);
    for (int i = 0; i < nv; ++i) {
        const float x = ld_one<ES>(v, e0 + i, bad);
        mx = fmax_nan(mx, x);
        if (x > best) {
            best = x;
            bidx = e_row0 + e0 + i;
        }
    }
}

// Loads the 8 elements of lane `lane` in block blk of a stage.
template <int ES>
static __device__ __forceinline__ int load_block8(const View &v, int blk, int lane, bool fast, float x[8], uint32_t &bad) {
    const int e = blk * kBlk + lane * 8;
    if (fast) {
        if (ES == 2) {
            uint4 w = *reinterpret_cast<const uint4 *>(v.s + 2 * e);
            x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x);
            x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
            x[4] = bf16_lo(w.z); x[5] = bf16_hi(w.z);
            x[6] = bf16_lo(w.w); x[7] = bf16_hi(w.w);
        } else {
            uint4 w0 = *reinterpret_cast<const uint4 *>(v.s + 4 * e);
            uint4 w1 = *reinterpret_cast<const uint4 *>(v.s + 4 * e + 16);
            x[0] = __uint_as_float(w0.x); x[1] = __uint_as_float(w0.y);
            x[2] = __uint_as_float(w0.z); x[3] = __uint_as_float(w0.w);
            x[4] = __uint_as_float(w1.x); x[5] = __uint_as_float(w1.y);
            x[6] = __uint_as_float(w1.z); x[7] = __uint_as_float(w1.w);
        }
        return max(0, min(8, v.cnt - e));
    }
    return load8<ES>(v, e, x, bad);
}

template <int ES, bool SMP>
static __device__ void consumer(const Params &P, Smem &S, const uint8_t *ring, int cw, int lane, uint32_t &bad) {
    int it = 0;      // stages consumed
    int uc = 0;      // units handed to the epilogue
    float best = -INFINITY;   // greedy: running max of this lane
    int bidx = -1;            // greedy: row index of its first occurrence
    float mx = -INFINITY;     // greedy: NaN-propagating max (non-finite detection)
    uint32_t pk = 0xff80ff80u;      // greedy bf16: per-half NaN-propagating max (starts at -inf)
    int glo = -1, ghi = -1;         // ... row index of the group that first set each half's max
    float Mw = -INFINITY;     // sampled: running max of this warp's blocks
    float Sw = 0.0f, Sc = 0.0f;   // sampled: compensated sum of 2^((z - Mw) c2)
    uint32_t epend = 0;       // greedy: children (lanes) not yet shown rejected
    float ethr = 0.0f;        // ... lane c: the logit of child c's draft token in this row
    int eidx = 0;             // ... lane c: b * R + child c
    constexpr int kPB = kPassBytes / ES / kBlk;                 // sampled: blocks per pass
    constexpr int kBPW = kPB / kConsumerWarps;                  // ... per warp
    static_assert(kPB % kConsumerWarps == 0, "pass blocks must split evenly over the consumer warps");
    while (true) {
        const int st = it % kStages;
        if (!wait_bar(P, S, &S.full[st], static_cast<uint32_t>((it / kStages) & 1))) break;
        const StageInfo &I = S.info[st];
        const uint4 hot = *reinterpret_cast<const uint4 *>(&S.info[st]);
        const int kind = static_cast<int>(hot.x & 15u);
        if (kind == kEnd) {
            // forward the end marker to every epilogue warp (the next kEpilogueWarps slots)
            bool ok = true;
            for (int q = 0; q < kEpilogueWarps && ok; ++q, ++uc) {
                const int slot = uc % kResSlots;
                if (uc >= kResSlots &&
                    !wait_bar(P, S, &S.res_empty[slot], static_cast<uint32_t>((uc / kResSlots - 1) & 1))) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    if (cw == 0) S.res[slot].kind = kEnd;
                    mbar_arrive(&S.res_full[slot]);
                }
            }
            ++it;
            break;
        }
        const uint8_t *stage = ring + static_cast<size_t>(st) * kStageBytes;
        const int last = static_cast<int>((hot.x >> 4) & 1u);
        const bool fast = ((hot.x >> 5) & 1u) != 0;
        const int cnt = static_cast<int>(hot.y);
        const int e0 = static_cast<int>(hot.z);
        const float c2 = SMP ? __uint_as_float(hot.w) : 0.0f;
        // unit identity, needed at the end of a unit (read before the stage is released)
        int b = 0, n = 0, j = 0, xtok = -1;
        float zx = 0.0f, qx = 0.0f, ux = 0.0f;
        if (last || kind == kB || c2 != 0.0f) {
            b = I.b;
            n = I.n;
            j = I.j;
            xtok = I.xtok;
            zx = I.zx;
            qx = I.qx;
            ux = I.ux;
        }
        // Fast stages are copied to registers and released before any arithmetic,
        // so the producer can refill the stage while this warp computes.
        auto release = [&]() {
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.empty[st]);
        };
        if (kind == kA && c2 == 0.0f) {
            // ---- greedy: running (max, first index) over 8-element groups
            if (hot.x & kFirstF) {
                // A child whose draft token's logit is beaten by any element of
                // this row is not the argmax: rejected, whatever the rest holds.
                const int nk = I.nk;
                epend = __ballot_sync(0xffffffffu, lane < nk);
                if (lane < nk) {
                    const int ko = I.kofs[lane];
                    const int bb = I.b, nn = I.n;
                    const int kid = kTree ? static_cast<int>(P.kid_list[P.kid_off[nn] + lane]) : nn + 1;
                    eidx = bb * P.R + kid;
                    if (ko >= 0) {
                        const uint8_t *pz = stage + kThrOff + 16 * lane + ko;
                        ethr = ES == 2 ? __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t *>(pz)) << 16)
                                       : *reinterpret_cast<const float *>(pz);
                    } else if (ko == -2) {
                        ethr = logit_global(P, in_row(P, bb, nn) * static_cast<size_t>(P.V) + I.ktok[lane]);
                    } else {
                        ethr = -INFINITY;
                    }
                }
            }
            const int ng = (cnt + 7) >> 3;
            if (ES == 2 && fast) {
                // bf16: packed per-half maxima with branch-free records, one pass at a time
                constexpr int kPG = kPassBytes / 16;   // groups per pass
                constexpr int kGPL = kPG / kConsumerLanes;
                static_assert(kPG % kConsumerLanes == 0, "pass must split evenly over the consumer lanes");
                for (int p0 = 0; p0 < ng; p0 += kPG) {
                    uint4 ra[kGPL];
#pragma unroll
                    for (int t = 0; t < kGPL; ++t) {
                        const int g = p0 + cw * 32 + lane + t * kConsumerLanes;
                        if (g < ng) ra[t] = *reinterpret_cast<const uint4 *>(stage + g * 16);
                    }
                    if (p0 + kPG >= ng) release();
#pragma unroll
                    for (int t = 0; t < kGPL; ++t) {
                        const int g = p0 + cw * 32 + lane + t * kConsumerLanes;
                        if (g < ng) {
                            const uint32_t a = bmax2_nan(bmax2_nan(ra[t].x, ra[t].y), bmax2_nan(ra[t].z, ra[t].w));
                            bf16x2_record(a, pk, e0 + 8 * g, glo, ghi);
                        }
                    }
                }
            } else if (fast) {
                constexpr int kPG = kPassBytes / (8 * ES);
                constexpr int kGPL = kPG / kConsumerLanes;
                static_assert(kPG % kConsumerLanes == 0, "pass must split evenly over the consumer lanes");
                for (int p0 = 0; p0 < ng; p0 += kPG) {
                    uint4 ra[kGPL], rc[kGPL];
#pragma unroll
                    for (int t = 0; t < kGPL; ++t) {
                        const int g = p0 + cw * 32 + lane + t * kConsumerLanes;
                        if (g < ng) {
                            ra[t] = *reinterpret_cast<const uint4 *>(stage + g * 8 * ES);
                            if (ES == 4) rc[t] = *reinterpret_cast<const uint4 *>(stage + g * 32 + 16);
                        }
                    }
                    if (p0 + kPG >= ng) release();
#pragma unroll
                    for (int t = 0; t < kGPL; ++t) {
                        const int g = p0 + cw * 32 + lane + t * kConsumerLanes;
                        if (g < ng) greedy_regs<ES>(ra[t], rc[t], e0 + 8 * g, best, bidx, mx);
                    }
                }
            } else {
                const View vz{stage + I.sh, I.gz, cnt, I.tail, I.sh == 0};
                for (int g = cw * 32 + lane; g < ng; g += kConsumerLanes)
                    group_step<ES>(vz, g, e0, false, best, bidx, mx, bad);
                release();
            }
            if (epend) {
                const float wm = warp_max_redux(fmaxf(best, fmaxf(bf16_lo(pk), bf16_hi(pk))));
                const uint32_t hit = __ballot_sync(0xffffffffu, ((epend >> lane) & 1u) && wm > ethr);
                if ((hit >> lane) & 1u) st_relaxed(P.early + eidx, 1u);
                epend &= ~hit;
            }
        } else if (SMP && kind == kA) {
            // ---- sampled: per 256-element block its max M and sum of 2^((z - M) c2)
            const View vz{stage + I.sh, I.gz, cnt, I.tail, I.sh == 0};
            const int nb = (cnt + kBlk - 1) / kBlk;
            const size_t rb = (static_cast<size_t>(b) * P.R + n) * P.nblk + e0 / kBlk;
            if (fast) {
              for (int p0 = 0; p0 < nb; p0 += kPB) {
                uint4 ra[kBPW], rc[kBPW];
#pragma unroll
                for (int t = 0; t < kBPW; ++t) {
                    const int blk = p0 + cw + t * kConsumerWarps;
                    if (blk < nb) {
                        const int e = blk * kBlk + lane * 8;
                        ra[t] = *reinterpret_cast<const uint4 *>(stage + e * ES);
                        if (ES == 4) rc[t] = *reinterpret_cast<const uint4 *>(stage + e * 4 + 16);
                    }
                }
                if (p0 + kPB >= nb) release();
                // One reference max M for all of this warp's blocks in the pass (any M at
                // or above a block's max works; it is stored with each block's sum).
                // cnt is a multiple of 8 here: a lane's 8 elements are all valid or none.
                float lm = -INFINITY;
#pragma unroll
                for (int t = 0; t < kBPW; ++t) {
                    const int blk = p0 + cw + t * kConsumerWarps;
                    if (blk < nb && blk * kBlk + lane * 8 < cnt)
                        lm = fmax_nan(lm, ES == 2 ? vmax8_bf16(ra[t]) : vmax8_f32(ra[t], rc[t]));
                }
                const float M = warp_max_redux(lm);
                const float nMc2 = neg_mc2(M, c2);
                const float2 c22 = make_float2(c2, c2), nm2 = make_float2(nMc2, nMc2);
                float sl[kBPW];   // this lane's partial of each of the warp's blocks
#pragma unroll
                for (int t = 0; t < kBPW; ++t) {
                    const int blk = p0 + cw + t * kConsumerWarps;
                    float s = 0.0f;
                    if (blk < nb && blk * kBlk + lane * 8 < cnt) {
                        float x[8];
                        unpack8<ES>(ra[t], rc[t], x);
                        float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const float2 a = fma2(make_float2(x[2 * k], x[2 * k + 1]), c22, nm2);
                            const float2 wv = make_float2(ex2(a.x), ex2(a.y));
                            acc = (k == 0) ? wv : add2(acc, wv);
                        }
                        s = __fadd_rn(acc.x, acc.y);
                    }
                    sl[t] = s;
                }
                // block totals, scattered over the lanes: lane l holds block q(l)
                const float tb = warp_sum_scatter<kBPW>(sl, lane);
                constexpr int kGroup = 32 / kBPW;   // lanes holding the same block
                const int q = kBPW == 4 ? (((lane >> 4) & 1) * 2 + ((lane >> 3) & 1)) : ((lane >> 4) & 1);
                const int bq = p0 + cw + q * kConsumerWarps;
                if ((lane & (kGroup - 1)) == 0 && bq < nb) {
                    P.bmaxA[rb + bq] = M;
                    P.bsumA[rb + bq] = tb;
                }
                // the pass total: the block totals summed across the groups
                float pt = tb;
#pragma unroll
                for (int off = kGroup; off < 32; off <<= 1) pt = __fadd_rn(pt, __shfl_xor_sync(0xffffffffu, pt, off));
                if (p0 + cw < nb) fold_stats(M, pt, c2, Mw, Sw, Sc);
              }
            } else {
                for (int blk = cw; blk < nb; blk += kConsumerWarps) {
                    float x[8];
                    const int nv = load8<ES>(vz, blk * kBlk + lane * 8, x, bad);
                    float lm = -INFINITY;
                    for (int i = 0; i < nv; ++i) lm = fmax_nan(lm, x[i]);
                    const float M = warp_max_redux(lm);
                    const float nMc2 = neg_mc2(M, c2);
                    float w[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) w[i] = (i < nv) ? w_exp(x[i], nMc2, c2) : 0.0f;
                    const float sblk = warp_butterfly_sum(lane_sum8(w));
                    if (lane == 0) {
                        P.bmaxA[rb + blk] = M;
                        P.bsumA[rb + blk] = sblk;
                    }
                    fold_stats(M, __shfl_sync(0xffffffffu, sblk, 0), c2, Mw, Sw, Sc);
                }
                release();
            }
        } else if (SMP) {
            // ---- residual: per 256-element block the sum of max(0, p - q)
            const View vz{stage + I.sh, I.gz, cnt, I.tail, I.sh == 0};
            const View vq{stage + P.qoff + I.shq, I.gq, cnt, I.tailq, I.shq == 0};
            const float m_row = I.m, invS = I.invS;
            const int nb = (cnt + kBlk - 1) / kBlk;   // at most one block per warp
            const int blk = cw;
            float x[8], y[8];
            int nvz = 0;
            if (fast) {
                uint4 za, zc, qa, qc;
                if (blk < nb) {
                    const int e = blk * kBlk + lane * 8;
                    za = *reinterpret_cast<const uint4 *>(stage + e * ES);
                    if (ES == 4) zc = *reinterpret_cast<const uint4 *>(stage + e * 4 + 16);
                    qa = *reinterpret_cast<const uint4 *>(stage + P.qoff + e * 4);
                    qc = *reinterpret_cast<const uint4 *>(stage + P.qoff + e * 4 + 16);
                }
                release();
                if (blk < nb) {
                    nvz = max(0, min(8, cnt - (blk * kBlk + lane * 8)));
                    unpack8<ES>(za, zc, x);
                    unpack8<4>(qa, qc, y);
                }
            } else {
                uint32_t qbad = 0;
                if (blk < nb) {
                    nvz = load8<ES>(vz, blk * kBlk + lane * 8, x, bad);
                    load8<4>(vq, blk * kBlk + lane * 8, y, qbad);
                }
                release();
            }
            if (blk < nb) {
                const float nmc2 = neg_mc2(m_row, c2);
                float w[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) w[i] = (i < nvz) ? w_res(x[i], y[i], nmc2, c2, invS) : 0.0f;
                const float s = warp_butterfly_sum(lane_sum8(w));
                if (lane == 0) P.bsumB[static_cast<size_t>(b) * P.nblk + e0 / kBlk + blk] = s;
            }
        }
        ++it;
        if (last) {
            // hand the unit to the epilogue
            const int slot = uc % kResSlots;
            if (uc >= kResSlots && !wait_bar(P, S, &S.res_empty[slot], static_cast<uint32_t>((uc / kResSlots - 1) & 1)))
                break;
            float v = best;
            int g = bidx;
            float pv = -INFINITY;   // greedy bf16: packed-record candidate (value, group)
            int pgw = -1;
            if (kind == kA && c2 == 0.0f) {
                warp_cand(v, g);
                if (ES == 2) {
                    // packed records: the lane's max and the first group holding it, then
                    // the warp's winner (the epilogue finds its first element in memory,
                    // off the consumers' path)
                    const float mlo = bf16_lo(pk), mhi = bf16_hi(pk);
                    pv = fmaxf(mlo, mhi);
                    pgw = mlo > mhi ? glo : (mhi > mlo ? ghi : min(static_cast<unsigned>(glo), static_cast<unsigned>(ghi)));
                    if (!(pv > -INFINITY)) pgw = -1;
                    warp_cand(pv, pgw);
                }
                mx = fmax_nan(mx, fmax_nan(bf16_lo(pk), bf16_hi(pk)));
                mx = fmax_nan(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                mx = fmax_nan(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmax_nan(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                mx = fmax_nan(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                mx = fmax_nan(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                // NaN or +inf seen by this warp (a warp that saw no element keeps -inf)
                if (lane == 0 && (mx != mx || mx == INFINITY)) set_status(P, SPEC_STATUS_NONFINITE);
            }
            if (lane == 0) {
                ResSlot &R = S.res[slot];
                if (kind == kA && c2 != 0.0f) {
                    R.v[cw] = Mw;
                    R.s[cw] = __fadd_rn(Sw, Sc);
                } else {
                    R.v[cw] = v;
                    R.idx[cw] = g;
                    R.s[cw] = pv;
                    R.pg[cw] = pgw;
                }
                if (cw == 0) {
                    R.kind = kind;
                    R.b = b;
                    R.n = n;
                    R.j = j;
                    R.c2 = c2;
                    R.xtok = xtok;
                    R.zx = zx;
                    R.qx = qx;
                    R.ux = ux;
                }
                mbar_arrive(&S.res_full[slot]);
            }
            ++uc;
            best = -INFINITY;
            bidx = -1;
            mx = -INFINITY;
            pk = 0xff80ff80u;
            glo = -1;
            ghi = -1;
            Mw = -INFINITY;
            Sw = 0.0f;
            Sc = 0.0f;
            epend = 0;
        }
    }
    if (lane == 0 && cw == 0) S.consumed = it;
}

template <bool SMP>
static __device__ void epilogue(const Params &P, Smem &S, int e, int lane) {
    int uc = e;   // this warp takes units e, e + kEpilogueWarps, ...
    while (true) {
        const int slot = uc % kResSlots;
        if (!wait_bar(P, S, &S.res_full[slot], static_cast<uint32_t>((uc / kResSlots) & 1))) break;
        const ResSlot &R = S.res[slot];
        const int kind = R.kind;
        if (kind == kEnd) break;
        const int b = R.b, n = R.n, j = R.j;
        const float c2 = R.c2;
        const int xtok = R.xtok;
        const float zx = R.zx, qx = R.qx, ux = R.ux;
        float v = lane < kConsumerWarps ? R.v[lane] : -INFINITY;
        int grp = lane < kConsumerWarps ? R.idx[lane] : -1;
        const float sw = lane < kConsumerWarps ? R.s[lane] : 0.0f;
        int pgr = lane < kConsumerWarps ? R.pg[lane] : -1;
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.res_empty[slot]);
        uc += kEpilogueWarps;
        int draw_row = -1;        // an inverse-CDF draw this warp makes for request b: the bonus token
        bool draw_res = false;    // (p of the last row) or the residual token (max(0, p - q) of row n)
        if (kind == kA) {
            const bool greedy = !SMP || (c2 == 0.0f);
            float um = 0.0f;
            tf uS = tf_of(0.0f);
            if (greedy) {
                warp_cand(v, grp);
                if (P.esize == 2) {
                    // packed records: the winning group's first element equal to its max
                    float pv = (lane < kConsumerWarps) ? sw : -INFINITY;
                    warp_cand(pv, pgr);
                    int pidx = -1;
                    if (pgr >= 0 && pgr + 8 <= P.V) {
                        const uint4 w = __ldg(reinterpret_cast<const uint4 *>(
                            P.logits + (in_row(P, b, n) * static_cast<size_t>(P.V) + pgr) * 2));
                        int i = 7;
                        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                        for (int q = 3; q >= 0; --q) {
                            if (bf16_hi(ww[q]) == pv) i = 2 * q + 1;
                            if (bf16_lo(ww[q]) == pv) i = 2 * q;
                        }
                        pidx = pgr + i;
                    }
                    cand_merge(v, grp, pv, pidx);
                }
            } else {
                // combine the consumer warps' (M_w, S_w) into the unit's (m, S)
                um = warp_max(v);
                tf t = tf_of(0.0f);
                if (lane < kConsumerWarps && sw != 0.0f) t = tf_prod(sw, ex2(__fmul_rn(__fsub_rn(v, um), c2)));
                uS = warp_sum_tf(t);
            }
            const size_t ri = static_cast<size_t>(b) * P.R + n;
            bool resolve_now = true;
            if (P.ns > 1) {
                uint32_t old = 0;
                if (lane == 0) {
                    Partial pr;
                    pr.v = greedy ? v : um;
                    pr.idx = grp;
                    pr.sh = uS.h;
                    pr.sl = uS.l;
                    P.partial[ri * P.ns + j] = pr;
                    // acq_rel: publishes the partial and the consumers' block data
                    old = atom_add_acqrel(P.row_ctr + ri, 1u);
                }
                old = __shfl_sync(0xffffffffu, old, 0) + 1u;
                // The last split in resolves the row.  (Splits of a row found dead
                // are never streamed, so such a row never completes: nothing needs it.)
                resolve_now = old == static_cast<uint32_t>(P.ns);
                if (resolve_now) {
                    __syncwarp();   // the whole warp reads the partials after lane 0's acquire
                    if (greedy) {
                        v = -INFINITY;
                        grp = -1;
                        for (int q = lane; q < P.ns; q += 32) {
                            const Partial *pp = P.partial + ri * P.ns + q;
                            cand_merge(v, grp, __ldcg(&pp->v), __ldcg(&pp->idx));
                        }
                        warp_cand(v, grp);
                    } else {
                        float lm = -INFINITY;
                        for (int q = lane; q < P.ns; q += 32) lm = fmaxf(lm, __ldcg(&P.partial[ri * P.ns + q].v));
                        um = warp_max(lm);
                        tf t = tf_of(0.0f);
                        for (int q = lane; q < P.ns; q += 32) {
                            const float4 w = __ldcg(reinterpret_cast<const float4 *>(P.partial + ri * P.ns + q));
                            if (w.z != 0.0f) t = tf_add(t, tf_mulf(tf{w.z, w.w}, ex2(__fmul_rn(__fsub_rn(w.x, um), c2))));
                        }
                        uS = warp_sum_tf(t);
                    }
                }
            }
            if (resolve_now) {
                resolve_row<SMP>(P, b, n, greedy, c2, grp, v, um, uS, xtok, zx, qx, ux, lane);
                draw_row = finish_row<SMP>(P, S, e, b, n, greedy, lane);
            }
        } else if (SMP) {
            // B unit: the last chunk of a request's residual draws the token
            uint32_t old = 0;
            // acq_rel: publishes this chunk's residual block sums; the last chunk's
            // acquire sees every chunk's (the warp then reads them after a warp sync)
            if (lane == 0) old = atom_add_acqrel(P.res_ctr + b, 1u);
            old = __shfl_sync(0xffffffffu, old, 0);
            if (old == static_cast<uint32_t>(P.ncb - 1)) {
                __syncwarp();
                draw_row = n;
                draw_res = true;
            }
        }
        if (SMP && draw_row >= 0) {
            const float u = __ldg(P.u_sample + in_row(P, b, draw_row));
            const int t = sample_row(P, b, draw_row, draw_res, u, lane);
            if (lane == 0) P.out_tokens[static_cast<size_t>(b) * (P.D + 1) + draw_row] = t;
        }
    }
}

};  // struct Dev

// --------------------------------------------------------------- kernel --
template <int ES, bool SMP, int MODE>
__global__ void __maxnreg__(128) verify_kernel(const __grid_constant__ Params P) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    Smem &S = *reinterpret_cast<Smem *>(smem_raw);
    uint8_t *ring = smem_raw + ((sizeof(Smem) + 127) & ~static_cast<size_t>(127));
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    uint32_t bad = 0;

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&S.full[i], 1);
            mbar_init(&S.empty[i], kConsumerWarps);
        }
        for (int i = 0; i < kResSlots; ++i) {
            mbar_init(&S.res_full[i], kConsumerWarps);
            mbar_init(&S.res_empty[i], 1);
        }
        S.abort_flag = 0;
        S.issued = 0;
        S.consumed = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // Every block of this grid is resident from the start, so the next kernel
    // may begin launching at once; nothing here touches global memory before
    // the previous kernel in the stream has completed.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __syncthreads();

    if (warp == 0) Dev<MODE>::template producer<ES, SMP>(P, S, ring, lane);
    else if (warp <= kEpilogueWarps) Dev<MODE>::template epilogue<SMP>(P, S, warp - 1, lane);
    else Dev<MODE>::template consumer<ES, SMP>(P, S, ring, warp - 1 - kEpilogueWarps, lane, bad);

    bad = __any_sync(0xffffffffu, bad != 0);
    if (lane == 0 && bad) set_status(P, SPEC_STATUS_NONFINITE);
    __syncthreads();
    if (tid == 0) {
        if (*reinterpret_cast<volatile int *>(&S.abort_flag)) {
            // Let copies still in flight land before the block's memory is reused.
            for (int it = S.consumed; it < S.issued; ++it) {
                uint64_t *bar = &S.full[it % kStages];
                unsigned long long t0 = globaltimer();
                while (!mbar_try_wait(bar, static_cast<uint32_t>((it / kStages) & 1)))
                    if (globaltimer() - t0 > kWaitLimitNs) break;
            }
        }
        uint32_t old = atom_add_acqrel(P.ctrl + 1, 1u);
        S.last_flag = (old == gridDim.x - 1);
    }
    __syncthreads();
    if (S.last_flag) {
        // every other block has finished with the counters: clear them for the next call
        for (uint32_t i = tid; i < P.reset_words; i += kThreads) P.reset_base[i] = 0u;
    }
}

// ------------------------------------------------------------ slot fix-up --
// Ragged chains: request b's slots are packed at cu[b] + b .. cu[b+1] + b (its
// drafts plus one); one warp per request keeps j <= num_accepted[b].
__global__ void fixup_ragged_kernel(int64_t *slots, int B, const int32_t *cu, int total, const int32_t *num_acc,
                                    int64_t pad) {
    const int w = static_cast<int>((blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (w >= B) return;
    int lo = __ldg(cu + w), hi = __ldg(cu + w + 1);
    lo = min(max(lo, 0), total);
    hi = min(max(hi, lo), total);
    const int a = __ldg(num_acc + w);
    int64_t *sb = slots + static_cast<size_t>(lo) + w;
    for (int j = lane; j <= hi - lo; j += 32)
        if (j > a) sb[j] = pad;
}

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

void clear_error() { g_err[0] = 0; }

spec_status_t fail(spec_status_t s, const char *fmt, const char *detail) {
    snprintf(g_err, sizeof g_err, fmt, detail);
    return s;
}

struct Layout {
    size_t stats, reset, reset_bytes, ctrl, req_mask, row_ctr, rowstate, req_ctr, req_state, res_ctr, early;
    size_t rowstat, partial, bmaxA, bsumA, bsumB, total;
    int esub, nsub, esb, ecb, qoff, ncb, nblk;
};

size_t up256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

bool make_layout(int B, int R, int V, spec_dtype_t dtype, Layout &L) {
    if (B < 1 || R < 1 || R > kMaxRows || V < 1 || V >= (1 << 30)) return false;
    if (dtype != SPEC_BF16 && dtype != SPEC_FP32) return false;
    const int es = dtype == SPEC_BF16 ? 2 : 4;
    // stages of a row balanced in size, each a whole number of 256-element blocks
    const int emax = kSubBytes / es;
    L.nsub = (V + emax - 1) / emax;
    L.esub = (((V + L.nsub - 1) / L.nsub) + kBlk - 1) / kBlk * kBlk;
    L.esb = kConsumerWarps * kBlk;   // one 256-element block per consumer warp
    static_assert(kConsumerWarps * kBlk * (4 + 4) + 64 <= kSubBytes + 128, "B stage does not fit");
    L.ecb = L.esb * kSubPerB;
    L.qoff = ((L.esb * es + 16) + 15) & ~15;
    L.ncb = (V + L.ecb - 1) / L.ecb;
    L.nblk = (V + kBlk - 1) / kBlk;
    const size_t BR = static_cast<size_t>(B) * R;
    size_t off = 0;
    L.stats = off;
    off = up256(off + 64);
    L.reset = off;
    L.ctrl = off;
    off += 32 * 4;
    L.req_mask = off;
    off += static_cast<size_t>(B) * 8;
    L.row_ctr = off;
    off += BR * 4;
    L.rowstate = off;
    off += BR * 4;
    L.req_ctr = off;
    off += static_cast<size_t>(B) * 4;
    L.req_state = off;
    off += static_cast<size_t>(B) * 4;
    L.res_ctr = off;
    off += static_cast<size_t>(B) * 4;
    L.early = off;
    off += BR * 4;
    off = up256(off);
    L.reset_bytes = off - L.reset;
    L.rowstat = off;
    off = up256(off + BR * sizeof(RowStat));
    L.partial = off;
    off = up256(off + BR * L.nsub * sizeof(Partial));
    L.bmaxA = off;
    off = up256(off + BR * L.nblk * 4);
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

constexpr size_t kSmemBytes = ((sizeof(Smem) + 127) & ~static_cast<size_t>(127)) +
                              static_cast<size_t>(kStages) * kStageBytes;
static_assert(kSmemBytes <= 227 * 1024, "shared memory of one block exceeds the sm_103 limit");

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
        // every instantiation: (element size 2 / 4) x (greedy-only / sampled) per mode
        // (padded chains, ragged chains), and greedy-only trees; even q are bf16
        const void *kernels[10] = {
            reinterpret_cast<const void *>(verify_kernel<2, false, 0>), reinterpret_cast<const void *>(verify_kernel<4, false, 0>),
            reinterpret_cast<const void *>(verify_kernel<2, true, 0>), reinterpret_cast<const void *>(verify_kernel<4, true, 0>),
            reinterpret_cast<const void *>(verify_kernel<2, false, 1>), reinterpret_cast<const void *>(verify_kernel<4, false, 1>),
            reinterpret_cast<const void *>(verify_kernel<2, true, 1>), reinterpret_cast<const void *>(verify_kernel<4, true, 1>),
            reinterpret_cast<const void *>(verify_kernel<2, false, 2>), reinterpret_cast<const void *>(verify_kernel<4, false, 2>)};
        for (int q = 0; q < 10 && e == cudaSuccess; ++q) {
            e = cudaFuncSetAttribute(kernels[q], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(kSmemBytes));
            int nb = 0;
            if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kernels[q], kThreads, kSmemBytes);
            if (e == cudaSuccess && (q < 2 || nb < D.blocks_per_sm[q & 1])) D.blocks_per_sm[q & 1] = nb;
        }
        if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "kernel setup: %s", cudaGetErrorString(e));
        if (D.blocks_per_sm[0] < 1 || D.blocks_per_sm[1] < 1) {
            cudaFuncAttributes fa;
            memset(&fa, 0, sizeof fa);
            cudaFuncGetAttributes(&fa, verify_kernel<2, true, 0>);
            char buf[200];
            snprintf(buf, sizeof buf, " (%d registers, max %d threads, %zu B static + %zu B dynamic shared, %d threads)",
                     fa.numRegs, fa.maxThreadsPerBlock, fa.sharedSizeBytes, kSmemBytes, kThreads);
            return fail(SPEC_ERR_UNSUPPORTED, "the verify kernel does not fit on this device%s", buf);
        }
        D.ok = 1;
    }
    out = &D;
    return SPEC_OK;
}

spec_status_t require_sm103(int *sms) {
    DeviceInfo *D = nullptr;
    spec_status_t st = device_info(D);
    if (st == SPEC_OK && sms) *sms = D->sms;
    return st;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Process-wide tuning and test settings (spec_set_tuning, spec_set_wait_limit_ns),
// read once per call when the launch is set up.
std::atomic<int> g_tune_splits{0};
std::atomic<int> g_tune_ahead{0};
std::atomic<int> g_tune_path{0};   // 0: automatic; 1: persistent only; 2: automatic plus greedy chains on clusters

bool chain_cluster_allowed() { return g_tune_path.load(std::memory_order_relaxed) != 1; }
int tuning_path() { return g_tune_path.load(std::memory_order_relaxed); }
std::atomic<unsigned long long> g_wait_ns{kWaitLimitNs};

unsigned long long wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }

// Splits per row: whole rows when the batch gives every SM about two rows,
// otherwise finer splits (down to one 16 KiB stage) so small batches still
// spread over the GPU.  A split count set by spec_set_tuning overrides it.
int choose_splits(int rows_total, int nsub, int sms) {
    int ns = (2 * sms + rows_total - 1) / rows_total;
    const int forced = g_tune_splits.load(std::memory_order_relaxed);
    if (forced > 0) ns = forced;
    if (ns < 1) ns = 1;
    if (ns > nsub) ns = nsub;
    return ns;
}

// Stages the producer keeps in flight: the whole ring, unless spec_set_tuning
// asked for fewer (2..ring size: fewer stages in flight let a row that turns
// out not to be needed stop sooner).
int choose_ahead() {
    const int forced = g_tune_ahead.load(std::memory_order_relaxed);
    return (forced >= 2 && forced <= kStages) ? forced : kStages;
}

// Launch with programmatic stream serialisation: the kernel's blocks may be
// scheduled while the kernel before it in the stream drains (each block waits,
// griddepcontrol.wait, before its first global memory access), so the launch
// and the blocks' start-up overlap the previous kernel's tail.
template <typename K>
static cudaError_t launch_serialised(K kernel, dim3 grid, cudaStream_t st, const Params &P) {
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, P);
}

// clear_counters: zero the layout's counter region on `stream` just before the
// launch, after every host check has passed (the no-alloc entry point's static
// scratch keeps whatever the previous call left).
spec_status_t launch_verify(Params &P, spec_dtype_t dtype, void *workspace, size_t ws_bytes, void *stream,
                            bool clear_counters = false) {
    Layout L;
    if (!make_layout(P.B, P.R, P.V, dtype, L)) return fail(SPEC_ERR_INVALID_ARG, "invalid sizes%s");
    if (!workspace || ws_bytes < L.total)
        return fail(SPEC_ERR_INVALID_ARG, "workspace missing or smaller than spec_workspace_bytes()%s");
    if (!aligned16(workspace)) return fail(SPEC_ERR_INVALID_ARG, "workspace must be 16-byte aligned%s");
    DeviceInfo *D = nullptr;
    spec_status_t s = device_info(D);
    if (s != SPEC_OK) return s;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    P.stats = reinterpret_cast<unsigned long long *>(ws + L.stats);
    P.ctrl = reinterpret_cast<uint32_t *>(ws + L.ctrl);
    P.row_ctr = reinterpret_cast<uint32_t *>(ws + L.row_ctr);
    P.rowstate = reinterpret_cast<uint32_t *>(ws + L.rowstate);
    P.req_ctr = reinterpret_cast<uint32_t *>(ws + L.req_ctr);
    P.req_state = reinterpret_cast<uint32_t *>(ws + L.req_state);
    P.res_ctr = reinterpret_cast<uint32_t *>(ws + L.res_ctr);
    P.early = reinterpret_cast<uint32_t *>(ws + L.early);
    P.req_mask = reinterpret_cast<unsigned long long *>(ws + L.req_mask);
    P.mask_mode = P.R <= 64;
    P.reset_base = reinterpret_cast<uint32_t *>(ws + L.reset);
    P.reset_words = static_cast<uint32_t>(L.reset_bytes / 4);
    P.rowstat = reinterpret_cast<RowStat *>(ws + L.rowstat);
    P.partial = reinterpret_cast<Partial *>(ws + L.partial);
    P.bmaxA = reinterpret_cast<float *>(ws + L.bmaxA);
    P.bsumA = reinterpret_cast<float *>(ws + L.bsumA);
    P.bsumB = reinterpret_cast<float *>(ws + L.bsumB);
    P.esize = dtype == SPEC_BF16 ? 2 : 4;
    P.esub = L.esub;
    P.nsub = L.nsub;
    P.esb = L.esb;
    P.ecb = L.ecb;
    P.qoff = L.qoff;
    P.ncb = L.ncb;
    P.nblk = L.nblk;
    // rows actually present (ragged chains: one more than the drafts per request)
    const long long rows_total = P.cu ? static_cast<long long>(P.total_drafts) + P.B : static_cast<long long>(P.B) * P.R;
    int ns = choose_splits(rows_total > (1 << 30) ? (1 << 30) : static_cast<int>(rows_total), L.nsub, D->sms);
    P.sps = (L.nsub + ns - 1) / ns;
    P.ahead = choose_ahead();
    P.wait_ns = wait_limit_ns();
    P.ns = (L.nsub + P.sps - 1) / P.sps;
    // units span the padded (node, request, split) space; ragged requests' missing
    // nodes are dropped by the producer without work
    const long long ua = static_cast<long long>(P.B) * P.R * P.ns;
    const long long ub = P.q ? static_cast<long long>(P.B) * L.ncb : 0;
    if (ua + ub >= (1ll << 31) - (1 << 20)) return fail(SPEC_ERR_INVALID_ARG, "batch too large%s");
    P.units_a = static_cast<int>(ua);
    P.units_total = static_cast<int>(ua + ub);
    const size_t zrows = static_cast<size_t>(rows_total);
    const size_t qrows = P.cu ? static_cast<size_t>(P.total_drafts) : static_cast<size_t>(P.B) * (P.R - 1);
    P.logits_end = reinterpret_cast<unsigned long long>(P.logits) + zrows * static_cast<size_t>(P.V) * P.esize;
    P.q_end = P.q ? reinterpret_cast<unsigned long long>(P.q) + qrows * static_cast<size_t>(P.V) * 4 : 0;
    long long grid = static_cast<long long>(D->sms) * D->blocks_per_sm[dtype == SPEC_BF16 ? 0 : 1];
    if (grid > P.units_total) grid = P.units_total;
    if (grid < 1) grid = 1;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (clear_counters) {
        const cudaError_t ec = cudaMemsetAsync(ws + L.reset, 0, L.reset_bytes, st);
        if (ec != cudaSuccess) return fail(SPEC_ERR_CUDA, "clearing the workspace counters: %s", cudaGetErrorString(ec));
    }
    if (!P.cu && !P.q && !P.temperature) {
        // greedy padded chains and greedy trees: the persistent cluster kernel
        GreedyClusterArgs A;
        memset(&A, 0, sizeof A);
        A.logits = P.logits;
        A.dtype = dtype;
        A.tokens = P.tokens;
        A.parent = P.tree ? P.parent : nullptr;
        A.B = P.B;
        A.R = P.R;
        A.V = P.V;
        A.D = P.D;
        A.out_tokens = P.out_tokens;
        A.out_count = P.out_count;
        A.out_path = P.out_path;
        A.slots = P.slots;
        A.pad = P.pad;
        A.status = P.status;
        A.stats = P.stats;
        A.ctr = P.ctrl;
        A.rmask = P.req_mask;
        A.dmask = reinterpret_cast<unsigned long long *>(ws + L.row_ctr);   // B words: R >= 2 rows of 4 bytes each
        A.fin = P.req_ctr;
        A.rowstate = P.rowstate;
        A.reset_base = P.reset_base;
        A.reset_words = static_cast<int>(P.reset_words);
        bool launched = false;
        const spec_status_t gs = launch_greedy_cluster(A, stream, launched);
        if (gs != SPEC_OK || launched) return gs;
    }
    // Calls without temperatures are greedy only: a leaner instantiation without
    // the sampling and residual code.
    const dim3 g3(static_cast<unsigned>(grid));
    const bool bf = dtype == SPEC_BF16;
    cudaError_t e = cudaSuccess;
    if (P.tree) {
        if (bf) e = launch_serialised(verify_kernel<2, false, 2>, g3, st, P);
        else e = launch_serialised(verify_kernel<4, false, 2>, g3, st, P);
    } else if (P.cu) {
        if (P.q || P.temperature) {
            if (bf) e = launch_serialised(verify_kernel<2, true, 1>, g3, st, P);
            else e = launch_serialised(verify_kernel<4, true, 1>, g3, st, P);
        } else {
            if (bf) e = launch_serialised(verify_kernel<2, false, 1>, g3, st, P);
            else e = launch_serialised(verify_kernel<4, false, 1>, g3, st, P);
        }
    } else if (P.q || P.temperature) {
        if (bf) e = launch_serialised(verify_kernel<2, true, 0>, g3, st, P);
        else e = launch_serialised(verify_kernel<4, true, 0>, g3, st, P);
    } else {
        if (bf) e = launch_serialised(verify_kernel<2, false, 0>, g3, st, P);
        else e = launch_serialised(verify_kernel<4, false, 0>, g3, st, P);
    }
    if (e == cudaSuccess) e = cudaGetLastError();
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

    Layout L;
    if (!make_layout(B, rows, V, dtype, L)) return 0;
    return L.total;
}

extern "C" spec_status_t spec_workspace_init(void *workspace, size_t bytes, void *stream) {
    if (!workspace) return fail(SPEC_ERR_INVALID_ARG, "workspace is NULL%s");
    cudaError_t e = cudaMemsetAsync(workspace, 0, bytes, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "cudaMemsetAsync: %s", cudaGetErrorString(e));
    return SPEC_OK;
}

namespace sv {
spec_status_t verify_chain_common(const void *target_logits, spec_dtype_t dtype, const float *draft_probs,
                                  const int32_t *draft_tokens, const float *temperature, const float *u_accept,
                                  const float *u_sample, int B, int k, int V, int32_t *out_tokens,
                                  int32_t *out_num_accepted, int64_t *slot_mapping, int64_t padding_slot_id,
                                  int32_t *d_status, void *workspace, size_t workspace_bytes, void *stream) {
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
    if (!make_layout(B, k + 1, V, dtype, L)) return fail(SPEC_ERR_INVALID_ARG, "invalid sizes%s");
    if (!workspace || workspace_bytes < L.total)
        return fail(SPEC_ERR_INVALID_ARG, "workspace missing or smaller than spec_workspace_bytes()%s");
    if (!aligned16(workspace)) return fail(SPEC_ERR_INVALID_ARG, "workspace must be 16-byte aligned%s");
    // a sampled batch whose per-request clusters fit on the GPU at once: one
    // cluster per request (greedy-only batches stream best on the persistent
    // kernel, which skips rows whose drafts are already known rejected)
    if (chain_cluster_allowed() && draft_probs) {
        const int C = chain_cluster_size(B, k, V, dtype == SPEC_BF16 ? 2 : 4);
        if (C > 0)
            return launch_chain_cluster(target_logits, dtype, draft_probs, draft_tokens, temperature, u_accept,
                                        u_sample, B, k, V, out_tokens, out_num_accepted, slot_mapping,
                                        padding_slot_id, d_status, workspace, C, stream);
    }
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
    P.slots = slot_mapping;
    P.pad = padding_slot_id;
    P.B = B;
    P.R = k + 1;
    P.V = V;
    P.D = k;
    P.tree = 0;
    return launch_verify(P, dtype, workspace, workspace_bytes, stream);
}
}  // namespace sv

extern "C" spec_status_t spec_verify_chain(const void *target_logits, spec_dtype_t dtype, const float *draft_probs,
                                           const int32_t *draft_tokens, const float *temperature,
                                           const float *u_accept, const float *u_sample, int B, int k, int V,
                                           int32_t *out_tokens, int32_t *out_num_accepted, int32_t *d_status,
                                           void *workspace, size_t workspace_bytes, void *stream) {
    return sv::verify_chain_common(target_logits, dtype, draft_probs, draft_tokens, temperature, u_accept, u_sample,
                                   B, k, V, out_tokens, out_num_accepted, nullptr, 0, d_status, workspace,
                                   workspace_bytes, stream);
}

extern "C" spec_status_t spec_verify_chain_fused(const void *target_logits, spec_dtype_t dtype,
                                                 const float *draft_probs, const int32_t *draft_tokens,
                                                 const float *temperature, const float *u_accept,
                                                 const float *u_sample, int B, int k, int V, int32_t *out_tokens,
                                                 int32_t *out_num_accepted, int64_t *slot_mapping,
                                                 int64_t padding_slot_id, int32_t *d_status, void *workspace,
                                                 size_t workspace_bytes, void *stream) {
    if (!slot_mapping) return sv::fail(SPEC_ERR_INVALID_ARG, "slot_mapping is NULL%s");
    return sv::verify_chain_common(target_logits, dtype, draft_probs, draft_tokens, temperature, u_accept, u_sample,
                                   B, k, V, out_tokens, out_num_accepted, slot_mapping, padding_slot_id, d_status,
                                   workspace, workspace_bytes, stream);
}

namespace sv {
spec_status_t verify_chain_ragged_common(const void *target_logits, spec_dtype_t dtype, const float *draft_probs,
                                         const int32_t *draft_tokens, const int32_t *cu_num_draft_tokens,
                                         int total_drafts, const float *temperature, const float *u_accept,
                                         const float *u_sample, int B, int max_k, int V, int32_t *out_tokens,
                                         int32_t *out_num_accepted, int64_t *slot_mapping, int64_t padding_slot_id,
                                         int32_t *d_status, void *workspace, size_t workspace_bytes, void *stream) {
    g_err[0] = 0;
    if (dtype != SPEC_BF16 && dtype != SPEC_FP32) return fail(SPEC_ERR_INVALID_ARG, "unknown dtype%s");
    if (B < 1 || max_k < 0 || max_k > kMaxRows - 1 || V < 1 || V >= (1 << 30) || total_drafts < 0 ||
        static_cast<long long>(total_drafts) > static_cast<long long>(B) * max_k)
        return fail(SPEC_ERR_INVALID_ARG,
                    "sizes out of range (1<=B, 0<=max_k<=255, 1<=V<2^30, 0<=total_drafts<=B*max_k)%s");
    if (!target_logits || !cu_num_draft_tokens || !out_tokens || !out_num_accepted ||
        (total_drafts > 0 && !draft_tokens))
        return fail(SPEC_ERR_INVALID_ARG, "a required pointer is NULL%s");
    // with no drafts at all, sampled requests need only temperature and u_sample
    const bool sampled = draft_probs || u_accept || u_sample || temperature;
    if (sampled && (!u_sample || !temperature || (total_drafts > 0 && (!draft_probs || !u_accept))))
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
    P.slots = slot_mapping;
    P.pad = padding_slot_id;
    P.B = B;
    P.R = max_k + 1;
    P.V = V;
    P.D = max_k;
    P.tree = 0;
    P.cu = cu_num_draft_tokens;
    P.total_drafts = total_drafts;
    return launch_verify(P, dtype, workspace, workspace_bytes, stream);
}
}  // namespace sv

extern "C" spec_status_t spec_verify_chain_ragged(const void *target_logits, spec_dtype_t dtype,
                                                  const float *draft_probs, const int32_t *draft_tokens,
                                                  const int32_t *cu_num_draft_tokens, int total_drafts,
                                                  const float *temperature, const float *u_accept,
                                                  const float *u_sample, int B, int max_k, int V,
                                                  int32_t *out_tokens, int32_t *out_num_accepted, int32_t *d_status,
                                                  void *workspace, size_t workspace_bytes, void *stream) {
    return sv::verify_chain_ragged_common(target_logits, dtype, draft_probs, draft_tokens, cu_num_draft_tokens,
                                          total_drafts, temperature, u_accept, u_sample, B, max_k, V, out_tokens,
                                          out_num_accepted, nullptr, 0, d_status, workspace, workspace_bytes, stream);
}

extern "C" spec_status_t spec_verify_chain_ragged_fused(
    const void *target_logits, spec_dtype_t dtype, const float *draft_probs, const int32_t *draft_tokens,
    const int32_t *cu_num_draft_tokens, int total_drafts, const float *temperature, const float *u_accept,
    const float *u_sample, int B, int max_k, int V, int32_t *out_tokens, int32_t *out_num_accepted,
    int64_t *slot_mapping, int64_t padding_slot_id, int32_t *d_status, void *workspace, size_t workspace_bytes,
    void *stream) {
    if (!slot_mapping) return sv::fail(SPEC_ERR_INVALID_ARG, "slot_mapping is NULL%s");
    return sv::verify_chain_ragged_common(target_logits, dtype, draft_probs, draft_tokens, cu_num_draft_tokens,
                                          total_drafts, temperature, u_accept, u_sample, B, max_k, V, out_tokens,
                                          out_num_accepted, slot_mapping, padding_slot_id, d_status, workspace,
                                          workspace_bytes, stream);
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
    // children lists, in node order (counting sort by parent)
    int cnt[kMaxRows + 1] = {0};
    for (int n = 1; n <= N; ++n) ++cnt[parent[n]];
    int off = 0;
    for (int n = 0; n <= N; ++n) {
        P.kid_off[n] = static_cast<uint8_t>(off);
        off += cnt[n];
        cnt[n] = P.kid_off[n];
    }
    P.kid_off[N + 1] = static_cast<uint8_t>(off);
    for (int n = 1; n <= N; ++n) P.kid_list[cnt[parent[n]]++] = static_cast<uint8_t>(n);
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

extern "C" spec_status_t spec_fixup_slots_ragged(int64_t *slot_mapping, int B, const int32_t *cu_num_draft_tokens,
                                                 int total_drafts, const int32_t *num_accepted,
                                                 int64_t padding_slot_id, void *stream) {
    g_err[0] = 0;
    if (B < 0 || total_drafts < 0) return fail(SPEC_ERR_INVALID_ARG, "negative size%s");
    if (B == 0) return SPEC_OK;
    if (!slot_mapping || !cu_num_draft_tokens || !num_accepted)
        return fail(SPEC_ERR_INVALID_ARG, "a required pointer is NULL%s");
    const long long threads = static_cast<long long>(B) * 32;
    fixup_ragged_kernel<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        slot_mapping, B, cu_num_draft_tokens, total_drafts, num_accepted, padding_slot_id);
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

extern "C" unsigned long long spec_set_wait_limit_ns(unsigned long long ns) {
    return g_wait_ns.exchange(ns, std::memory_order_relaxed);
}

extern "C" spec_status_t spec_set_tuning(int splits, int ahead, int path) {
    g_err[0] = 0;
    if (splits < 0 || ahead < 0 || (ahead != 0 && (ahead < 2 || ahead > kStages)) || path < 0 || path > 2)
        return fail(SPEC_ERR_INVALID_ARG, "need splits >= 0, ahead 0 or in [2, 3], path 0, 1 or 2%s");
    g_tune_splits.store(splits, std::memory_order_relaxed);
    g_tune_ahead.store(ahead, std::memory_order_relaxed);
    g_tune_path.store(path, std::memory_order_relaxed);
    return SPEC_OK;
}

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
    if (!make_layout(B, k + 1, V, dtype, L)) return fail(SPEC_ERR_INVALID_ARG, "invalid sizes%s");
    if (L.total > kNoAllocScratchBytes) {
        char buf[160];
        snprintf(buf, sizeof buf, "these sizes need %zu bytes of scratch; the static scratch holds %zu bytes",
                 L.total, kNoAllocScratchBytes);
        return fail(SPEC_ERR_INVALID_ARG, "%s (use spec_verify_chain with a workspace)", buf);
    }
    // The device must be supported before the scratch is looked up (a device
    // that is not 10.3 reports SPEC_ERR_UNSUPPORTED, not a symbol-lookup error).
    spec_status_t s = require_sm103(nullptr);
    if (s != SPEC_OK) return s;
    uint8_t *scratch = nullptr;
    s = noalloc_scratch_ptr(scratch);
    if (s != SPEC_OK) return s;
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
    // The same dispatch as spec_verify_chain (the cluster kernel needs no scratch).
    if (chain_cluster_allowed() && draft_probs) {
        const int C = chain_cluster_size(B, k, V, dtype == SPEC_BF16 ? 2 : 4);
        if (C > 0)
            return launch_chain_cluster(target_logits, dtype, draft_probs, draft_tokens, temperature, u_accept,
                                        u_sample, B, k, V, out_tokens, out_num_accepted, nullptr, 0, d_status,
                                        nullptr, C, stream);
    }
    // The scratch keeps whatever the previous call left; launch_verify clears
    // this layout's counter region once every check has passed.
    return launch_verify(P, dtype, scratch, kNoAllocScratchBytes, stream, true);
}
