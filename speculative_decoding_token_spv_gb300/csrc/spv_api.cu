// spv_api.cu -- the C ABI of libspv (declared in include/spv.h): argument
// checks on the host, workspace sizing, and dispatch to the kernels.
#include "spv.h"
#include "spv_internal.h"

#include <cmath>
#include <cstdint>
#include <cstring>

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned256(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }
int elem_bytes(spv_dtype d) { return d == SPV_F32 ? 4 : 2; }
bool dtype_ok(spv_dtype d) { return d == SPV_F32 || d == SPV_BF16; }

// Every logit index must fit an int; the largest row offset must fit size_t.
bool sizes_ok(int B, int rows_per_seq, int V)
{
    if (B < 1 || rows_per_seq < 1 || V < 2) return false;
    const double total = static_cast<double>(B) * rows_per_seq * V;
    return total < 9.0e15;
}

spv_status cuda_status(cudaError_t e) { return e == cudaSuccess ? SPV_OK : SPV_ERR_CUDA; }

}  // namespace

extern "C" {

size_t spv_chain_workspace_bytes(int B, int gamma, int V)
{
    if (B < 1 || gamma < 1 || gamma > SPV_MAX_GAMMA || V < 2) return 0;
    return spv::chain_ws_bytes(B, gamma, V);
}

size_t spv_greedy_workspace_bytes(int B, int gamma, int V)
{
    if (B < 1 || gamma < 1 || gamma > SPV_MAX_GAMMA || V < 2) return 0;
    return spv::greedy_ws_bytes(B, gamma, V);
}

size_t spv_fanout_workspace_bytes(int B, int K, int V, int max_fanout)
{
    if (B < 1 || K < 0 || K + 1 > SPV_MAX_FANOUT_ROWS || V < 2 || max_fanout < 0 || max_fanout > SPV_MAX_FANOUT)
        return 0;
    return spv::fanout_ws_bytes(B, K + 1, V, max_fanout);
}

}  // extern "C"

namespace spv {

spv_status check_chain_args(const ChainArgs &a)
{
    if (!dtype_ok(a.dtype) || !a.target_logits || !a.draft_tokens || !a.accept_count || !a.out_tokens)
        return SPV_ERR_INVALID_ARG;
    if (a.gamma < 1 || a.gamma > SPV_MAX_GAMMA || !sizes_ok(a.B, 2 * a.gamma + 1, a.V)) return SPV_ERR_INVALID_ARG;
    if (!(a.temperature >= 0.0f) || std::isinf(a.temperature)) return SPV_ERR_INVALID_ARG;
    if (a.temperature > 0.0f) {
        if (!a.draft_logits || !a.r || !a.sample_keys) return SPV_ERR_INVALID_ARG;
        if (!(1.0f / a.temperature < INFINITY)) return SPV_ERR_INVALID_ARG;  // T too small to invert
    }
    return SPV_OK;
}

size_t chain_call_ws_bytes(const ChainArgs &a)
{
    return a.temperature == 0.0f ? greedy_ws_bytes(a.B, a.gamma, a.V) : chain_ws_bytes(a.B, a.gamma, a.V);
}

ChainLaunch chain_launch(const ChainArgs &a, void *ws)
{
    ChainLaunch L{};
    L.target = a.target_logits;
    L.draft = a.draft_logits;
    L.dtype = a.dtype == SPV_F32 ? 0 : 1;
    L.tokens = a.draft_tokens;
    L.r = a.r;
    L.keys = a.sample_keys;
    L.B = a.B;
    L.gamma = a.gamma;
    L.V = a.V;
    L.T = a.temperature;
    L.accept_count = a.accept_count;
    L.out_tokens = a.out_tokens;
    L.out_pq = a.out_pq;
    L.out_Z = a.out_resid_norm;
    L.row_status = a.row_status;
    L.ws = ws;
    const bool greedy = a.temperature == 0.0f;
    const bool rows16 = (static_cast<size_t>(a.V) * elem_bytes(a.dtype)) % 16 == 0;
    L.tma = rows16 && aligned16(a.target_logits) && (greedy || aligned16(a.draft_logits));
    return L;
}

cudaError_t launch_chain_or_greedy(const ChainLaunch &L, cudaStream_t st)
{
    return L.T == 0.0f ? launch_greedy(L, st) : launch_chain(L, st);
}

}  // namespace spv

namespace {

spv_status verify_chain_impl(const spv::ChainArgs &a, const int32_t *cache_ids, const int32_t *fanout,
                             int32_t *cache_slot, void *workspace, size_t workspace_bytes, void *stream,
                             float sag_C = 0.0f)
{
    const spv_status chk = spv::check_chain_args(a);
    if (chk != SPV_OK) return chk;
    if (!workspace || !aligned256(workspace)) return SPV_ERR_INVALID_ARG;
    if (workspace_bytes < spv::chain_call_ws_bytes(a)) return SPV_ERR_INVALID_ARG;
    if (cache_ids || fanout || cache_slot) {
        if (!cache_ids || !fanout || !cache_slot) return SPV_ERR_INVALID_ARG;
        for (int k = 0; k <= a.gamma; ++k)
            if (fanout[k] < 0 || fanout[k] > SPV_MAX_FANOUT) return SPV_ERR_INVALID_ARG;
    }
    spv::ChainLaunch L = spv::chain_launch(a, workspace);
    L.cache_ids = cache_ids;
    L.cache_fanout = fanout;
    L.cache_slot = cache_slot;
    L.sag = sag_C > 0.0f ? 1 : 0;
    L.sag_C = sag_C;
    return cuda_status(spv::launch_chain_or_greedy(L, static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

spv_status spv_verify_chain(const void *target_logits, const void *draft_logits, spv_dtype dtype,
                            const int32_t *draft_tokens, const float *r, const uint64_t *sample_keys, int B,
                            int gamma, int V, float temperature, int32_t *accept_count, int32_t *out_tokens,
                            float *out_pq, float *out_resid_norm, int32_t *row_status, void *workspace,
                            size_t workspace_bytes, void *stream)
{
    const spv::ChainArgs a{target_logits, draft_logits, dtype, draft_tokens, r, sample_keys, B, gamma, V,
                           temperature, accept_count, out_tokens, out_pq, out_resid_norm, row_status};
    return verify_chain_impl(a, nullptr, nullptr, nullptr, workspace, workspace_bytes, stream);
}

spv_status spv_verify_chain_cached(const void *target_logits, const void *draft_logits, spv_dtype dtype,
                                   const int32_t *draft_tokens, const float *r, const uint64_t *sample_keys,
                                   int B, int gamma, int V, float temperature, int32_t *accept_count,
                                   int32_t *out_tokens, float *out_pq, float *out_resid_norm, int32_t *row_status,
                                   const int32_t *cache_ids, const int32_t *fanout, int32_t *cache_slot,
                                   void *workspace, size_t workspace_bytes, void *stream)
{
    if (!cache_ids || !fanout || !cache_slot) return SPV_ERR_INVALID_ARG;
    const spv::ChainArgs a{target_logits, draft_logits, dtype, draft_tokens, r, sample_keys, B, gamma, V,
                           temperature, accept_count, out_tokens, out_pq, out_resid_norm, row_status};
    return verify_chain_impl(a, cache_ids, fanout, cache_slot, workspace, workspace_bytes, stream);
}

spv_status spv_verify_chain_saguaro(const void *target_logits, const void *draft_logits, spv_dtype dtype,
                                    const int32_t *draft_tokens, const float *r, const uint64_t *sample_keys, int B,
                                    int gamma, int V, float temperature, const int32_t *cache_ids,
                                    const int32_t *fanout, float C, int32_t *accept_count, int32_t *out_tokens,
                                    float *out_pq, float *out_resid_norm, int32_t *row_status, int32_t *cache_slot,
                                    void *workspace, size_t workspace_bytes, void *stream)
{
    if (!cache_ids || !fanout || !cache_slot) return SPV_ERR_INVALID_ARG;
    if (!(C > 0.0f) || std::isinf(C) || !(1.0f / C > 0.0f) || std::isinf(1.0f / C)) return SPV_ERR_INVALID_ARG;
    if (spv::blocks_per_row(V) > 1024) return SPV_ERR_UNSUPPORTED;  // V > 1,048,576
    const spv::ChainArgs a{target_logits, draft_logits, dtype, draft_tokens, r, sample_keys, B, gamma, V,
                           temperature, accept_count, out_tokens, out_pq, out_resid_norm, row_status};
    return verify_chain_impl(a, cache_ids, fanout, cache_slot, workspace, workspace_bytes, stream, C);
}

size_t spv_tree_workspace_bytes(int B, int N, int V)
{
    if (B < 1 || N < 1 || N > SPV_MAX_TREE_NODES || V < 2) return 0;
    return spv::tree_ws_bytes(B, N, V);
}

spv_status spv_verify_tree(const void *target_logits, const void *draft_logits, spv_dtype dtype, const int32_t *parent,
                           const int32_t *tokens, const float *r, const uint64_t *sample_keys, int B, int N, int V,
                           float temperature, int32_t *accept_count, int32_t *out_tokens, int32_t *out_nodes,
                           int32_t *row_status, void *workspace, size_t workspace_bytes, void *stream)
{
    if (!dtype_ok(dtype) || !target_logits || !parent || !tokens || !accept_count || !out_tokens || !workspace)
        return SPV_ERR_INVALID_ARG;
    if (N < 1 || N > SPV_MAX_TREE_NODES || !sizes_ok(B, 2 * N, V)) return SPV_ERR_INVALID_ARG;
    if (!(temperature >= 0.0f) || std::isinf(temperature)) return SPV_ERR_INVALID_ARG;
    if (!aligned256(workspace) || workspace_bytes < spv::tree_ws_bytes(B, N, V)) return SPV_ERR_INVALID_ARG;
    const bool greedy = temperature == 0.0f;
    if (!greedy && (!draft_logits || !r || !sample_keys)) return SPV_ERR_INVALID_ARG;
    if (!greedy && !(1.0f / temperature < INFINITY)) return SPV_ERR_INVALID_ARG;
    spv::TreeLaunch L{};
    L.target = target_logits;
    L.draft = draft_logits;
    L.dtype = dtype == SPV_F32 ? 0 : 1;
    L.parent = parent;
    L.tokens = tokens;
    L.r = r;
    L.keys = sample_keys;
    L.B = B;
    L.N = N;
    L.V = V;
    L.T = temperature;
    L.accept_count = accept_count;
    L.out_tokens = out_tokens;
    L.out_nodes = out_nodes;
    L.row_status = row_status;
    L.ws = workspace;
    const bool rows16 = (static_cast<size_t>(V) * elem_bytes(dtype)) % 16 == 0;
    L.tma = rows16 && aligned16(target_logits) && (greedy || aligned16(draft_logits));
    return cuda_status(spv::launch_tree(L, static_cast<cudaStream_t>(stream)));
}

size_t spv_filtered_workspace_bytes(int B, int gamma, int V)
{
    if (B < 1 || gamma < 1 || gamma > SPV_MAX_GAMMA || V < 2) return 0;
    return spv::filtered_ws_bytes(B, gamma, V);
}

spv_status spv_verify_chain_filtered(const void *target_logits, const void *draft_logits, spv_dtype dtype,
                                     const int32_t *draft_tokens, const float *r, const uint64_t *sample_keys,
                                     int B, int gamma, int V, float temperature, int top_k, float top_p,
                                     int32_t *accept_count, int32_t *out_tokens, float *out_pq,
                                     float *out_resid_norm, int32_t *row_status, void *workspace,
                                     size_t workspace_bytes, void *stream)
{
    if (!dtype_ok(dtype) || !target_logits || !draft_tokens || !accept_count || !out_tokens || !workspace)
        return SPV_ERR_INVALID_ARG;
    if (gamma < 1 || gamma > SPV_MAX_GAMMA || !sizes_ok(B, 2 * gamma + 1, V)) return SPV_ERR_INVALID_ARG;
    if (!(temperature >= 0.0f) || std::isinf(temperature)) return SPV_ERR_INVALID_ARG;
    if (top_k < 1 || top_k > SPV_MAX_TOP_K || !(top_p > 0.0f) || !(top_p <= 1.0f)) return SPV_ERR_INVALID_ARG;
    if (!aligned256(workspace)) return SPV_ERR_INVALID_ARG;
    const bool greedy = temperature == 0.0f;
    const size_t need = greedy ? spv::greedy_ws_bytes(B, gamma, V) : spv::filtered_ws_bytes(B, gamma, V);
    if (workspace_bytes < need) return SPV_ERR_INVALID_ARG;
    if (!greedy && (!draft_logits || !r || !sample_keys)) return SPV_ERR_INVALID_ARG;
    if (!greedy && !(1.0f / temperature < INFINITY)) return SPV_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * (2 * gamma + 1) * spv::chunks_per_row(V) > 0x7fffffffLL) return SPV_ERR_UNSUPPORTED;

    spv::ChainLaunch L{};
    L.target = target_logits;
    L.draft = draft_logits;
    L.dtype = dtype == SPV_F32 ? 0 : 1;
    L.tokens = draft_tokens;
    L.r = r;
    L.keys = sample_keys;
    L.B = B;
    L.gamma = gamma;
    L.V = V;
    L.T = temperature;
    L.top_k = top_k;
    L.top_p = top_p;
    L.accept_count = accept_count;
    L.out_tokens = out_tokens;
    L.out_pq = out_pq;
    L.out_Z = out_resid_norm;
    L.row_status = row_status;
    L.ws = workspace;
    const bool rows16 = (static_cast<size_t>(V) * elem_bytes(dtype)) % 16 == 0;
    L.tma = rows16 && aligned16(target_logits) && (greedy || aligned16(draft_logits));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return cuda_status(greedy ? spv::launch_greedy(L, st) : spv::launch_filtered(L, st));
}

spv_status spv_verify_greedy(const void *target_logits, spv_dtype dtype, const int32_t *draft_tokens, int B,
                             int gamma, int V, int32_t *accept_count, int32_t *out_tokens, int32_t *row_status,
                             void *workspace, size_t workspace_bytes, void *stream)
{
    if (!dtype_ok(dtype) || !target_logits || !draft_tokens || !accept_count || !out_tokens || !workspace)
        return SPV_ERR_INVALID_ARG;
    if (gamma < 1 || gamma > SPV_MAX_GAMMA || !sizes_ok(B, gamma + 1, V)) return SPV_ERR_INVALID_ARG;
    if (!aligned256(workspace) || workspace_bytes < spv::greedy_ws_bytes(B, gamma, V)) return SPV_ERR_INVALID_ARG;
    spv::ChainLaunch L{};
    L.target = target_logits;
    L.dtype = dtype == SPV_F32 ? 0 : 1;
    L.tokens = draft_tokens;
    L.B = B;
    L.gamma = gamma;
    L.V = V;
    L.accept_count = accept_count;
    L.out_tokens = out_tokens;
    L.row_status = row_status;
    L.ws = workspace;
    L.tma = (static_cast<size_t>(V) * elem_bytes(dtype)) % 16 == 0 && aligned16(target_logits);
    return cuda_status(spv::launch_greedy(L, static_cast<cudaStream_t>(stream)));
}

spv_status spv_fanout_topk(const void *draft_logits, spv_dtype dtype, const int32_t *exclude, const int32_t *fanout,
                           int B, int K, int V, int32_t *out_ids, int32_t *row_status, void *workspace,
                           size_t workspace_bytes, void *stream)
{
    if (!dtype_ok(dtype) || !draft_logits || !exclude || !fanout || !out_ids || !workspace)
        return SPV_ERR_INVALID_ARG;
    if (K < 0 || K + 1 > SPV_MAX_FANOUT_ROWS || !sizes_ok(B, K + 1, V)) return SPV_ERR_INVALID_ARG;
    if (spv::blocks_per_row(V) > 8 * 32 * 4) return SPV_ERR_UNSUPPORTED;  // V > 1,048,576
    spv::FanoutLaunch L{};
    L.K1 = K + 1;
    L.off[0] = 0;
    L.Fmax = 0;
    for (int k = 0; k <= K; ++k) {
        const int f = fanout[k];
        if (f < 0 || f > SPV_MAX_FANOUT || f > V - 1) return SPV_ERR_INVALID_ARG;
        L.F[k] = f;
        L.off[k + 1] = L.off[k] + f;
        if (f > L.Fmax) L.Fmax = f;
    }
    if (!aligned256(workspace) || workspace_bytes < spv::fanout_ws_bytes(B, K + 1, V, L.Fmax))
        return SPV_ERR_INVALID_ARG;
    L.draft = draft_logits;
    L.dtype = dtype == SPV_F32 ? 0 : 1;
    L.exclude = exclude;
    L.B = B;
    L.V = V;
    L.out_ids = out_ids;
    L.row_status = row_status;
    L.ws = workspace;
    L.tma = (static_cast<size_t>(V) * elem_bytes(dtype)) % 16 == 0 && aligned16(draft_logits);
    return cuda_status(spv::launch_fanout(L, static_cast<cudaStream_t>(stream)));
}

double spv_fanout_size(int F0, double a, double r, int k)
{
    return static_cast<double>(F0) * std::pow(a, static_cast<double>(k) / (1.0 + r));
}

spv_status spv_fanout_sizes(int F0, double a, double r, int K, int V, int32_t *out)
{
    if (!out || F0 < 0 || K < 0 || K + 1 > SPV_MAX_FANOUT_ROWS || V < 2) return SPV_ERR_INVALID_ARG;
    if (!(a > 0.0) || std::isinf(a) || !(r > -1.0) || std::isinf(r)) return SPV_ERR_INVALID_ARG;
    for (int k = 0; k <= K; ++k) {
        const double f = spv_fanout_size(F0, a, r, k);  // >= 0: F0 >= 0, a > 0
        const double n = std::floor(f + 0.5);           // half away from zero
        out[k] = static_cast<int32_t>(n > V - 1 ? V - 1 : n);
    }
    return SPV_OK;
}

spv_status spv_selftest_timeout(void *workspace, size_t workspace_bytes, unsigned polls, void *stream)
{
    if (!workspace || !aligned256(workspace) || workspace_bytes < spv::WS_HEADER) return SPV_ERR_INVALID_ARG;
    if (polls < 1 || polls > (1u << 24)) return SPV_ERR_INVALID_ARG;
    return cuda_status(spv::launch_selftest_wait(workspace, polls, static_cast<cudaStream_t>(stream)));
}

spv_status spv_workspace_status(const void *workspace, void *stream)
{
    if (!workspace) return SPV_ERR_INVALID_ARG;
    unsigned word = 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return SPV_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return SPV_ERR_CUDA;
    return word == 0 ? SPV_OK : static_cast<spv_status>(word);
}

const char *spv_status_string(spv_status s)
{
    switch (s) {
    case SPV_OK: return "SPV_OK";
    case SPV_ERR_INVALID_ARG: return "SPV_ERR_INVALID_ARG";
    case SPV_ERR_CUDA: return "SPV_ERR_CUDA";
    case SPV_ERR_UNSUPPORTED: return "SPV_ERR_UNSUPPORTED";
    case SPV_ERR_BAD_ROW: return "SPV_ERR_BAD_ROW";
    case SPV_ERR_TIMEOUT: return "SPV_ERR_TIMEOUT";
    }
    return "SPV_ERR_UNKNOWN";
}

}  // extern "C"
