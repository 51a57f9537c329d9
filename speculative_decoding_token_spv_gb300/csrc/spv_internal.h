// spv_internal.h -- host-side launch interface between spv_api.cu and the
// per-op kernel files.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "spv.h"

namespace spv {

// Workspace header: word 0 is the device error word (SPV_OK or
// SPV_ERR_TIMEOUT); sections start at multiples of 256 bytes.
constexpr size_t WS_HEADER = 256;
inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
inline int blocks_per_row(int V) { return (V + 1023) / 1024; }
inline int chunks_per_row(int V) { return (V + 8191) / 8192; }

struct ChainLaunch {
    const void *target, *draft;
    int dtype;  // 0 fp32, 1 bf16
    const int32_t *tokens;
    const float *r;
    const uint64_t *keys;
    int B, gamma, V;
    float T;
    int32_t *accept_count, *out_tokens;
    float *out_pq, *out_Z;
    int32_t *row_status;
    void *ws;
    bool tma;  // rows are 16-byte aligned and V * elem_bytes % 16 == 0
    // Optional speculation-cache lookup (null cache_ids: none).
    const int32_t *cache_ids;
    const int32_t *cache_fanout;  // host, gamma + 1 entries
    int32_t *cache_slot;
    // Top-k / top-p filter (spv_verify_chain_filtered only).
    int top_k;
    float top_p;
    // Saguaro sampling (spv_verify_chain_saguaro only): the cache lists are
    // the cached candidates whose draft probability was divided by sag_C.
    int sag;
    float sag_C;
};

struct TreeLaunch {
    const void *target, *draft;
    int dtype;
    const int32_t *parent, *tokens;
    const float *r;
    const uint64_t *keys;
    int B, N, V;
    float T;
    int32_t *accept_count, *out_tokens, *out_nodes, *row_status;
    void *ws;
    bool tma;
};

struct FanoutLaunch {
    const void *draft;
    int dtype;
    const int32_t *exclude;
    int F[64];
    int off[65];
    int Fmax;
    int B, K1, V;
    int32_t *out_ids, *row_status;
    void *ws;
    bool tma;
};

// The arguments spv_verify_chain shares with spv_verify_chain_noalloc.
struct ChainArgs {
    const void *target_logits, *draft_logits;
    spv_dtype dtype;
    const int32_t *draft_tokens;
    const float *r;
    const uint64_t *sample_keys;
    int B, gamma, V;
    float temperature;
    int32_t *accept_count, *out_tokens;
    float *out_pq, *out_resid_norm;
    int32_t *row_status;
};

// Host checks of those arguments (pointers, dtype, sizes, temperature):
// SPV_OK or the status the call returns before any launch.
spv_status check_chain_args(const ChainArgs &a);
// Scratch bytes the call needs (greedy layout at T == 0).
size_t chain_call_ws_bytes(const ChainArgs &a);
// The launch description of a checked call on scratch `ws` (no cache lookup,
// no Saguaro weights).
ChainLaunch chain_launch(const ChainArgs &a, void *ws);
// Enqueues the call: the greedy kernels at T == 0, else the chain kernels.
cudaError_t launch_chain_or_greedy(const ChainLaunch &L, cudaStream_t st);

size_t chain_ws_bytes(int B, int gamma, int V);
size_t greedy_ws_bytes(int B, int gamma, int V);
size_t fanout_ws_bytes(int B, int K1, int V, int Fmax);
size_t filtered_ws_bytes(int B, int gamma, int V);
size_t tree_ws_bytes(int B, int N, int V);

cudaError_t launch_chain(const ChainLaunch &L, cudaStream_t st);
cudaError_t launch_greedy(const ChainLaunch &L, cudaStream_t st);
cudaError_t launch_fanout(const FanoutLaunch &L, cudaStream_t st);
cudaError_t launch_filtered(const ChainLaunch &L, cudaStream_t st);
cudaError_t launch_selftest_wait(void *ws, unsigned polls, cudaStream_t st);
cudaError_t launch_tree(const TreeLaunch &L, cudaStream_t st);

}  // namespace spv
