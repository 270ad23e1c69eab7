// Host helpers shared by the translation units of libspecverify.
#pragma once

#include <stdint.h>

#include "spec_verify.h"

namespace sv {

// Clears the message spec_last_error() returns (at the start of a call).
void clear_error();

// Records the message (fmt with one %s for detail) for spec_last_error() and
// returns s.
spec_status_t fail(spec_status_t s, const char *fmt, const char *detail = "");

// SPEC_OK when the current device is compute capability 10.3; fills *sms with
// its SM count.
spec_status_t require_sm103(int *sms);

// Limit in nanoseconds of the kernels' waits on other blocks and warps
// (spec_set_wait_limit_ns); copies still in flight at a kernel's exit are
// always waited for with the default limit.
unsigned long long wait_limit_ns();

// Sampled (or mixed) chains in the padded layout whose per-request clusters all
// fit on the GPU at once go to the cluster kernel (chain_cluster.cu): the
// cluster size, or 0 for the persistent kernel.  spec_set_tuning can rule the
// cluster kernel out.
int chain_cluster_size(int B, int k, int V, int es);
bool chain_cluster_allowed();
// spec_set_tuning's path (0 automatic, 1 persistent only, 2 automatic plus
// greedy padded chains on the greedy cluster kernel).
int tuning_path();
spec_status_t launch_chain_cluster(const void *target_logits, spec_dtype_t dtype, const float *draft_probs,
                                   const int32_t *draft_tokens, const float *temperature, const float *u_accept,
                                   const float *u_sample, int B, int k, int V, int32_t *out_tokens,
                                   int32_t *out_num_accepted, int64_t *slot_mapping, int64_t padding_slot_id,
                                   int32_t *d_status, void *workspace, int C, void *stream);

// Greedy padded chains and greedy trees of at most 64 rows go to the
// persistent cluster kernel (greedy_cluster.cu) when its geometry fits; the
// workspace words are those of the persistent kernel's layout (its counter
// region, left zero again at exit).
struct GreedyClusterArgs {
    const void *logits;
    spec_dtype_t dtype;
    const int32_t *tokens;          // [B, R-1]
    const int16_t *parent;          // host [R] (trees) or null (chains)
    int B, R, V, D;
    int32_t *out_tokens, *out_count, *out_path;
    int64_t *slots;
    int64_t pad;
    int32_t *status;
    unsigned long long *stats;
    uint32_t *ctr;
    unsigned long long *rmask, *dmask;
    uint32_t *fin, *rowstate, *reset_base;
    int reset_words;
};
// launched: false (and SPEC_OK) when the call is not one the kernel takes.
spec_status_t launch_greedy_cluster(const GreedyClusterArgs &A, void *stream, bool &launched);

}  // namespace sv
