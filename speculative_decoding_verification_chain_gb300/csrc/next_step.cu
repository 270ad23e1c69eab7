// next_step.cu -- after verification: the next step's inputs and tree KV
// compaction, on sm_103a.
//
// What it computes (vLLM EAGLE walkthrough, "slot mapping and KV-cache
// management", which names the next-step helpers; EAGLE-3 review, "EAGLE-3
// inference" step 5: only the accepted path's KV is kept and drafting
// restarts from the confirmed prefix).  Readings, since the pages give names
// only: request b verified rows 0..k at sequence positions pos_b..pos_b+k; with
// a_b drafts accepted its next input is the token emitted last,
// out_tokens[b][a_b], at position pos_b + a_b + 1; the next step writes P_next
// rows at the positions that follow, each in the slot its block table gives;
// an EAGLE drafter reads the target's row of the last accepted position.  For
// a token tree, depth i of the accepted path must end where the chain keeps
// position i: the KV row of path node n_i moves from slot_mapping[b][n_i] to
// slot_mapping[b][i], every destination receiving its source's row as it was
// before the call.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "common.h"
#include "spec_verify.h"

namespace sv {
namespace ns {

constexpr int kPrepThreads = 256;
constexpr int kCompactThreads = 256;
constexpr int kGroup = 8;             // sources loaded before any of their destinations is stored
constexpr int kMaxPath = SPEC_MAX_ROWS;

struct PrepParams {
    const int32_t *out_tokens;   // [B, out_stride]
    const int32_t *num_accepted; // [B]
    const int32_t *positions;    // [B]
    const int32_t *block_table;  // [B, max_blocks]
    const int32_t *cu;           // [B+1] or null
    const uint8_t *hidden_in;    // [rows, row_bytes] or null
    uint8_t *hidden_out;         // [B, row_bytes]
    int32_t *next_token, *next_position, *last_row;
    int64_t *next_slots;         // [B, P_next]
    int32_t *status;
    int64_t row_bytes, pad;
    int out_stride, max_blocks, block_size, P_next, rows_per_req, hidden_vec;
};

// One block per request: the scalars, the P_next slots, then the hidden row
// (16-byte vectors when every row starts on a 16-byte boundary).
__global__ void __launch_bounds__(kPrepThreads) prepare_next_kernel(const __grid_constant__ PrepParams P) {
    const int b = blockIdx.x;
    int a = __ldg(P.num_accepted + b);
    int st = 0;
    // a at most the request's drafts (and inside out_tokens), so every row read stays in the request
    const int amax = min(P.out_stride - 1, P.cu ? __ldg(P.cu + b + 1) - __ldg(P.cu + b) : P.rows_per_req - 1);
    if (a < 0 || a > amax) {
        st |= SPEC_STATUS_BAD_OFFSETS;
        a = min(max(a, 0), max(amax, 0));
    }
    const long long np = static_cast<long long>(__ldg(P.positions + b)) + a + 1;
    const long long r = (P.cu ? static_cast<long long>(__ldg(P.cu + b)) + b
                              : static_cast<long long>(b) * P.rows_per_req) + a;
    if (threadIdx.x == 0) {
        P.next_token[b] = __ldg(P.out_tokens + static_cast<size_t>(b) * P.out_stride + a);
        P.next_position[b] = static_cast<int32_t>(np);
        if (P.last_row) P.last_row[b] = static_cast<int32_t>(r);
    }
    for (int j = threadIdx.x; j < P.P_next; j += kPrepThreads) {
        const long long pos = np + j;
        const long long blk = pos / P.block_size;
        int64_t slot = P.pad;
        if (pos >= 0 && blk < P.max_blocks) {
            const int32_t e = __ldg(P.block_table + static_cast<size_t>(b) * P.max_blocks + blk);
            if (e >= 0)
                slot = static_cast<int64_t>(e) * P.block_size + pos % P.block_size;
            else
                st |= SPEC_STATUS_SLOT_RANGE;
        } else {
            st |= SPEC_STATUS_SLOT_RANGE;
        }
        P.next_slots[static_cast<size_t>(b) * P.P_next + j] = slot;
    }
    if (P.hidden_in) {
        const uint8_t *src = P.hidden_in + static_cast<size_t>(r) * static_cast<size_t>(P.row_bytes);
        uint8_t *dst = P.hidden_out + static_cast<size_t>(b) * static_cast<size_t>(P.row_bytes);
        if (P.hidden_vec) {
            const long long nv = P.row_bytes / 16;
            for (long long i = threadIdx.x; i < nv; i += kPrepThreads)
                reinterpret_cast<uint4 *>(dst)[i] = __ldg(reinterpret_cast<const uint4 *>(src) + i);
        } else {
            for (long long i = threadIdx.x; i < P.row_bytes; i += kPrepThreads) dst[i] = __ldg(src + i);
        }
    }
    if (st && P.status) atomicOr(P.status, st);
}

struct CompactParams {
    uint8_t *kv;                  // [num_slots, row_bytes]
    const int64_t *slot_mapping;  // [B, slot_stride]
    const int32_t *path;          // [B, path_stride]
    const int32_t *out_len;       // [B]
    int32_t *status;
    int64_t num_slots, row_bytes;
    int slot_stride, path_stride;
};

// Blocks (b, x): request b, 16-byte columns [x * 256, x * 256 + 256) of the
// rows.  The copies of a request are taken in groups of kGroup depths: each
// thread loads its column of every source of the group, then stores them.
// Path node indices strictly increase (checked), so n_j >= j: a source of a
// later group is never the destination of an earlier one, and inside a group
// every load comes before every store, so each destination receives its
// source's row as it was before the call.
__global__ void __launch_bounds__(kCompactThreads) compact_kv_kernel(const __grid_constant__ CompactParams P) {
    __shared__ int64_t src_s[kMaxPath], dst_s[kMaxPath];
    __shared__ int ok_s;
    const int b = blockIdx.y;
    int L = __ldg(P.out_len + b);
    if (threadIdx.x == 0) ok_s = 1;
    __syncthreads();
    if (L < 1 || L > P.path_stride) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && P.status) atomicOr(P.status, SPEC_STATUS_BAD_OFFSETS);
        return;
    }
    const int32_t *path = P.path + static_cast<size_t>(b) * P.path_stride;
    const int64_t *slots = P.slot_mapping + static_cast<size_t>(b) * P.slot_stride;
    int st = 0;
    for (int i = threadIdx.x; i < L; i += kCompactThreads) {
        const int node = __ldg(path + i);
        const int prev = i > 0 ? __ldg(path + i - 1) : -1;
        src_s[i] = -1;
        dst_s[i] = -1;
        if (i == 0) {
            if (node != 0) ok_s = 0;
            continue;
        }
        if (node <= prev || node >= P.slot_stride || i >= P.slot_stride) {
            ok_s = 0;
            continue;
        }
        if (node == i) continue;
        const int64_t s = __ldg(slots + node), t = __ldg(slots + i);
        if (s < 0 || s >= P.num_slots || t < 0 || t >= P.num_slots) {
            st |= SPEC_STATUS_SLOT_RANGE;
            continue;
        }
        src_s[i] = s;
        dst_s[i] = t;
    }
    __syncthreads();
    const bool first = blockIdx.x == 0;
    if (!ok_s) {  // not a root-to-node path with increasing indices: the request is left alone
        if (threadIdx.x == 0 && first && P.status) atomicOr(P.status, SPEC_STATUS_BAD_OFFSETS);
        return;
    }
    if (st && first && P.status) atomicOr(P.status, st);
    const long long nv = P.row_bytes / 16;
    const long long col = static_cast<long long>(blockIdx.x) * kCompactThreads + threadIdx.x;
    if (col >= nv) return;
    for (int g0 = 1; g0 < L; g0 += kGroup) {
        uint4 v[kGroup];
#pragma unroll
        for (int j = 0; j < kGroup; ++j) {
            const int i = g0 + j;
            if (i < L && src_s[i] >= 0)
                v[j] = *reinterpret_cast<const uint4 *>(P.kv + static_cast<size_t>(src_s[i]) * P.row_bytes + col * 16);
        }
#pragma unroll
        for (int j = 0; j < kGroup; ++j) {
            const int i = g0 + j;
            if (i < L && src_s[i] >= 0)
                *reinterpret_cast<uint4 *>(P.kv + static_cast<size_t>(dst_s[i]) * P.row_bytes + col * 16) = v[j];
        }
    }
}

}  // namespace ns
}  // namespace sv

extern "C" spec_status_t spec_prepare_next_step(const int32_t *out_tokens, int out_stride,
                                                const int32_t *num_accepted, const int32_t *positions,
                                                const int32_t *block_table, int max_blocks, int block_size, int B,
                                                int P_next, int rows_per_req, const int32_t *cu_num_draft_tokens,
                                                const void *hidden_in, int64_t row_bytes, int64_t padding_slot_id,
                                                int32_t *next_token, int32_t *next_position, int64_t *next_slots,
                                                int32_t *last_row, void *hidden_out, int32_t *d_status,
                                                void *stream) {
    using namespace sv;
    clear_error();
    if (B < 0 || out_stride < 1 || max_blocks < 0 || block_size < 1 || P_next < 0)
        return fail(SPEC_ERR_INVALID_ARG, "need B >= 0, out_stride >= 1, max_blocks >= 0, block_size >= 1, P_next >= 0%s");
    if (!cu_num_draft_tokens && rows_per_req < 1)
        return fail(SPEC_ERR_INVALID_ARG, "rows_per_req must be >= 1 without cu_num_draft_tokens%s");
    if (B == 0) return SPEC_OK;
    if (!out_tokens || !num_accepted || !positions || !next_token || !next_position)
        return fail(SPEC_ERR_INVALID_ARG, "a required pointer is NULL%s");
    if (P_next > 0 && (!block_table || !next_slots))
        return fail(SPEC_ERR_INVALID_ARG, "block_table and next_slots are required when P_next > 0%s");
    if (hidden_in && (!hidden_out || row_bytes < 1))
        return fail(SPEC_ERR_INVALID_ARG, "hidden_out and row_bytes >= 1 are required with hidden_in%s");
    spec_status_t st = require_sm103(nullptr);
    if (st != SPEC_OK) return st;
    ns::PrepParams P;
    memset(&P, 0, sizeof P);
    P.out_tokens = out_tokens;
    P.num_accepted = num_accepted;
    P.positions = positions;
    P.block_table = block_table;
    P.cu = cu_num_draft_tokens;
    P.hidden_in = static_cast<const uint8_t *>(hidden_in);
    P.hidden_out = static_cast<uint8_t *>(hidden_out);
    P.next_token = next_token;
    P.next_position = next_position;
    P.last_row = last_row;
    P.next_slots = next_slots;
    P.status = d_status;
    P.row_bytes = row_bytes;
    P.pad = padding_slot_id;
    P.out_stride = out_stride;
    P.max_blocks = max_blocks;
    P.block_size = block_size;
    P.P_next = P_next;
    P.rows_per_req = rows_per_req;
    P.hidden_vec = hidden_in && row_bytes % 16 == 0 && reinterpret_cast<uintptr_t>(hidden_in) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(hidden_out) % 16 == 0;
    ns::prepare_next_kernel<<<static_cast<unsigned>(B), ns::kPrepThreads, 0, static_cast<cudaStream_t>(stream)>>>(P);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "next-step launch: %s", cudaGetErrorString(e));
    return SPEC_OK;
}

extern "C" spec_status_t spec_compact_tree_kv(void *kv, int64_t num_slots, int64_t row_bytes,
                                              const int64_t *slot_mapping, int slot_stride, const int32_t *path,
                                              int path_stride, const int32_t *out_len, int B, int32_t *d_status,
                                              void *stream) {
    using namespace sv;
    clear_error();
    if (B < 0 || num_slots < 0 || row_bytes < 16 || row_bytes % 16 != 0 || slot_stride < 1 || path_stride < 1 ||
        path_stride > ns::kMaxPath)
        return fail(SPEC_ERR_INVALID_ARG,
                    "need B >= 0, num_slots >= 0, row_bytes a positive multiple of 16, slot_stride >= 1, "
                    "1 <= path_stride <= 256%s");
    if (B == 0 || num_slots == 0) return SPEC_OK;
    if (!kv || !slot_mapping || !path || !out_len) return fail(SPEC_ERR_INVALID_ARG, "a required pointer is NULL%s");
    if (reinterpret_cast<uintptr_t>(kv) % 16 != 0) return fail(SPEC_ERR_INVALID_ARG, "kv must be 16-byte aligned%s");
    spec_status_t st = require_sm103(nullptr);
    if (st != SPEC_OK) return st;
    ns::CompactParams P;
    memset(&P, 0, sizeof P);
    P.kv = static_cast<uint8_t *>(kv);
    P.slot_mapping = slot_mapping;
    P.path = path;
    P.out_len = out_len;
    P.status = d_status;
    P.num_slots = num_slots;
    P.row_bytes = row_bytes;
    P.slot_stride = slot_stride;
    P.path_stride = path_stride;
    const long long nv = row_bytes / 16;
    const long long gx = (nv + ns::kCompactThreads - 1) / ns::kCompactThreads;
    if (gx > 0x7fffffffLL || B > 65535) return fail(SPEC_ERR_INVALID_ARG, "row_bytes or B too large for one launch%s");
    dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(B));
    ns::compact_kv_kernel<<<grid, ns::kCompactThreads, 0, static_cast<cudaStream_t>(stream)>>>(P);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SPEC_ERR_CUDA, "compaction launch: %s", cudaGetErrorString(e));
    return SPEC_OK;
}
