// spv_chain.cu -- chain verify (T > 0) and greedy verify (T = 0) kernels.
//
// Chain verify, "Speculative Decoding: How Draft-Model Parallelism Cuts LLM
// Inference Latency", section "The four-phase loop", steps 2-4:
//   one pass over the gamma+1 target rows and gamma draft rows of every
//   sequence computes, per 1024-logit sampler block, the block max m and
//   S = sum exp((z - m) / T).  The CTA that finishes a sequence's last work
//   item merges the blocks into row softmax statistics, runs the accept test
//   r_i q_i(x_i) <= p_i(x_i) for every draft token, finds the first
//   rejection with a warp ballot, and draws the emitted token: the bonus from
//   p_gamma, or the residual norm(max(0, p_k - q_k)) by rejection trials from
//   p_k (eight trials at a time, one per warp).  Draws use the two-level
//   exponential race over the per-block statistics plus a re-read of one
//   1024-logit block, so no row is read twice from HBM.
//
// Greedy verify, "Speculative Pipeline Decoding", streaming verification
// ("under greedy decoding we require an exact argmax match"): the same pass
// over the target rows keeps per-block (max, lowest argmax id); the finishing
// CTA compares each draft token with its row argmax.
#include "spv_internal.h"
#include "spv_stream.cuh"

#include <climits>

namespace spv {

// =====================================================================================
// Chain verify, T > 0
// =====================================================================================
struct ChainParams {
    long long total_items;
    int nc, nb, V;
    unsigned *counter;
    unsigned *err;
    const unsigned char *target, *draft;
    const int32_t *tokens;
    const float *r;
    const uint64_t *keys;
    int B, gamma, R;
    float invT, c2;  // 1/T and log2(e)/T
    int32_t *accept_count, *out_tokens;
    float *out_pq, *out_Z;
    int32_t *row_status;
    float2 *stats;   // [B*R*nb] (block max of z, sum exp((z - max)/T)); NaN max = bad block
    float *resid;    // [B*nb] residual block masses (direct draw / normaliser only)
};

struct ChainSmem {
    float M[2 * 32 + 1];  // row max of the raw logits
    float S[2 * 32 + 1];  // row sum exp((z - M)/T)
    int bad;
    int k;
    int trial_x[NCW];
    int trial_acc[NCW];
    int result;
    float Z;
};

template <int DT> struct ChainOp {
    using Params = ChainParams;
    using Smem = ChainSmem;
    static constexpr int EB = DType<DT>::BYTES;

    __device__ static __forceinline__ const unsigned char *row_of(const Params &P, int b, int rho)
    {
        if (rho <= P.gamma)
            return P.target + (static_cast<size_t>(b) * (P.gamma + 1) + rho) * static_cast<size_t>(P.V) * EB;
        return P.draft + (static_cast<size_t>(b) * P.gamma + (rho - P.gamma - 1)) * static_cast<size_t>(P.V) * EB;
    }
    __device__ static __forceinline__ const void *row_ptr(const Params &P, long long row)
    {
        const int b = static_cast<int>(row / P.R);
        return row_of(P, b, static_cast<int>(row - static_cast<long long>(b) * P.R));
    }
    __device__ static __forceinline__ int group(const Params &P, long long row) { return static_cast<int>(row / P.R); }
    __device__ static __forceinline__ int items_per_group(const Params &P) { return P.R * P.nc; }

    // Block statistics: m = max z (raw), s = sum exp((z - m) / T).
    __device__ static __forceinline__ void block(const Params &P, long long row, int beta, float v[32], int, int lane)
    {
        float m = -INFINITY;
#pragma unroll
        for (int e = 0; e < 32; ++e) m = fmaxf(m, v[e]);
        m = warp_max(m);
        const float mu = (m == -INFINITY) ? 0.f : m;
        float s = 0.f;
#pragma unroll
        for (int e = 0; e < 32; ++e) s += fast_exp2((v[e] - mu) * P.c2);
        s = warp_sum(s);
        if (lane == 0) {
            // NaN anywhere, or +inf (then inf - inf), makes s NaN.
            P.stats[row * P.nb + beta] = isnan(s) ? make_float2(__int_as_float(0x7fffffff), 0.f) : make_float2(m, s);
        }
    }

    __device__ static __forceinline__ float prob(const Params &P, const unsigned char *rowp, int x, float M, float S)
    {
        return expf((DType<DT>::load(rowp, x) - M) * P.invT) / S;
    }

    // Two-level exponential race drawing one id from softmax(row / T), using
    // the row's block statistics; one warp.  Returns the id.
    __device__ static int race_p(const Params &P, long long row, const unsigned char *rowp, float M, uint64_t key,
                                 uint32_t trial, uint32_t pos, int lane)
    {
        float best = -INFINITY;
        int bi = INT_MAX;
        for (int g = lane; 4 * g < P.nb; g += 32) {
            uint64_t w[4];
            philox_group(w, key, STREAM_BLOCK, trial, pos, static_cast<uint64_t>(g));
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int beta = 4 * g + e;
                if (beta < P.nb) {
                    const float2 st = __ldcg(&P.stats[row * P.nb + beta]);
                    const float sc = st.y > 0.f ? ((st.x - M) * P.invT + logf(st.y)) - log_expo(w[e]) : -INFINITY;
                    if (sc > best) {
                        best = sc;
                        bi = beta;
                    }
                }
            }
        }
        warp_argmax(best, bi);
        const float mb = __ldcg(&P.stats[row * P.nb + bi]).x;
        const int base = bi * G;
        const int cnt = min(G, P.V - base);
        best = -INFINITY;
        int bx = INT_MAX;
        for (int g = lane; 4 * g < cnt; g += 32) {
            uint64_t w[4];
            philox_group(w, key, STREAM_TOKEN, trial, pos, static_cast<uint64_t>(base >> 2) + g);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int x = base + 4 * g + e;
                if (x < P.V) {
                    const float z = DType<DT>::load(rowp, x);
                    const float sc = (z == -INFINITY) ? -INFINITY : (z - mb) * P.invT - log_expo(w[e]);
                    if (sc > best) {
                        best = sc;
                        bx = x;
                    }
                }
            }
        }
        warp_argmax(best, bx);
        return bx;
    }

    // Residual masses w = max(0, p - q) of one row pair, per block, into
    // P.resid; returns Z = sum w in sm.Z.  All consumer warps.
    __device__ static void residual_pass(const Params &P, int b, const unsigned char *tp, const unsigned char *dp,
                                         float Mt, float St, float Md, float Sd, Smem &sm, int warp, int lane)
    {
        const float it = 1.f / St, id = 1.f / Sd;
        for (int beta = warp; beta < P.nb; beta += NCW) {
            float part = 0.f;
            const int hi = min(P.V, (beta + 1) * G);
            for (int x = beta * G + lane; x < hi; x += 32) {
                const float p = expf((DType<DT>::load(tp, x) - Mt) * P.invT) * it;
                const float q = expf((DType<DT>::load(dp, x) - Md) * P.invT) * id;
                part += fmaxf(p - q, 0.f);
            }
            part = warp_sum(part);
            if (lane == 0) P.resid[static_cast<size_t>(b) * P.nb + beta] = part;
        }
        consumer_sync();
        if (warp == 0) {
            float z = 0.f;
            for (int beta = lane; beta < P.nb; beta += 32) z += __ldcg(&P.resid[static_cast<size_t>(b) * P.nb + beta]);
            z = warp_sum(z);
            if (lane == 0) sm.Z = z;
        }
        consumer_sync();
    }

    // Direct race over the residual (after the rejection trials all failed).
    __device__ static int race_resid(const Params &P, int b, const unsigned char *tp, const unsigned char *dp,
                                     float Mt, float St, float Md, float Sd, uint64_t key, uint32_t pos, int lane)
    {
        float best = -INFINITY;
        int bi = INT_MAX;
        for (int g = lane; 4 * g < P.nb; g += 32) {
            uint64_t w[4];
            philox_group(w, key, STREAM_FB_BLOCK, 0, pos, static_cast<uint64_t>(g));
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int beta = 4 * g + e;
                if (beta < P.nb) {
                    const float W = __ldcg(&P.resid[static_cast<size_t>(b) * P.nb + beta]);
                    const float sc = W > 0.f ? logf(W) - log_expo(w[e]) : -INFINITY;
                    if (sc > best) {
                        best = sc;
                        bi = beta;
                    }
                }
            }
        }
        warp_argmax(best, bi);
        const float it = 1.f / St, id = 1.f / Sd;
        const int base = bi * G, cnt = min(G, P.V - base);
        best = -INFINITY;
        int bx = INT_MAX;
        for (int g = lane; 4 * g < cnt; g += 32) {
            uint64_t w[4];
            philox_group(w, key, STREAM_FB_TOKEN, 0, pos, static_cast<uint64_t>(base >> 2) + g);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int x = base + 4 * g + e;
                if (x < P.V) {
                    const float p = expf((DType<DT>::load(tp, x) - Mt) * P.invT) * it;
                    const float q = expf((DType<DT>::load(dp, x) - Md) * P.invT) * id;
                    const float wx = fmaxf(p - q, 0.f);
                    const float sc = wx > 0.f ? logf(wx) - log_expo(w[e]) : -INFINITY;
                    if (sc > best) {
                        best = sc;
                        bx = x;
                    }
                }
            }
        }
        warp_argmax(best, bx);
        return bx;
    }

    __device__ static void finalize(const Params &P, int b, Smem &sm, int warp, int lane)
    {
        const int R = P.R, g = P.gamma;
        if (threadIdx.x == 0) sm.bad = 0;
        consumer_sync();
        // 1. Merge block statistics into row statistics (one warp per row).
        for (int rho = warp; rho < R; rho += NCW) {
            const float2 *st = P.stats + (static_cast<long long>(b) * R + rho) * P.nb;
            float m = -INFINITY;
            bool bad = false;
            for (int beta = lane; beta < P.nb; beta += 32) {
                const float2 v = __ldcg(&st[beta]);
                if (isnan(v.x)) bad = true;
                else m = fmaxf(m, v.x);
            }
            m = warp_max(m);
            bad = __any_sync(0xffffffffu, bad);
            float s = 0.f;
            if (!bad && m != -INFINITY) {
                for (int beta = lane; beta < P.nb; beta += 32) {
                    const float2 v = __ldcg(&st[beta]);
                    if (v.y > 0.f) s += v.y * expf((v.x - m) * P.invT);
                }
            }
            s = warp_sum(s);
            if (lane == 0) {
                sm.M[rho] = m;
                sm.S[rho] = s;
                if (bad || !(s > 0.f)) atomicOr(&sm.bad, 1);
            }
        }
        if (warp == 0 && lane < g) {
            const int x = P.tokens[static_cast<size_t>(b) * g + lane];
            if (x < 0 || x >= P.V) atomicOr(&sm.bad, 1);
        }
        consumer_sync();
        const uint64_t key = P.keys[b];
        if (sm.bad) {
            for (int i = threadIdx.x; i <= g; i += NCW * 32) P.out_tokens[static_cast<size_t>(b) * (g + 1) + i] = -1;
            if (P.out_pq)
                for (int i = threadIdx.x; i < 2 * g; i += NCW * 32)
                    P.out_pq[static_cast<size_t>(b) * 2 * g + i] = __int_as_float(0x7fffffff);
            if (threadIdx.x == 0) {
                P.accept_count[b] = -1;
                if (P.row_status) P.row_status[b] = STATUS_BAD_ROW;
                if (P.out_Z) P.out_Z[b] = __int_as_float(0x7fffffff);
                P.counter[b] = 0u;
            }
            consumer_sync();
            return;
        }
        // 2. Accept tests for every draft position; first rejection by ballot.
        if (warp == 0) {
            bool acc = false;
            if (lane < g) {
                const int x = P.tokens[static_cast<size_t>(b) * g + lane];
                const float p = prob(P, row_of(P, b, lane), x, sm.M[lane], sm.S[lane]);
                const float q = prob(P, row_of(P, b, g + 1 + lane), x, sm.M[g + 1 + lane], sm.S[g + 1 + lane]);
                const float rr = P.r[static_cast<size_t>(b) * g + lane];
                acc = (p > 0.f) && (rr * q <= p);
                if (P.out_pq) {
                    P.out_pq[(static_cast<size_t>(b) * g + lane) * 2] = p;
                    P.out_pq[(static_cast<size_t>(b) * g + lane) * 2 + 1] = q;
                }
            }
            const unsigned mask = __ballot_sync(0xffffffffu, acc);
            const unsigned all = (g == 32) ? 0xffffffffu : ((1u << g) - 1u);
            if (lane == 0) sm.k = ((mask & all) == all) ? g : (__ffs(~mask) - 1);
        }
        consumer_sync();
        const int k = sm.k;
        // 3. The emitted token.
        const unsigned char *tp = row_of(P, b, k);
        const long long trow = static_cast<long long>(b) * R + k;
        if (k == g) {
            if (warp == 0) {
                const int x = race_p(P, trow, tp, sm.M[k], key, 0u, static_cast<uint32_t>(g), lane);
                if (lane == 0) sm.result = x;
            }
            consumer_sync();
        } else {
            const unsigned char *dp = row_of(P, b, g + 1 + k);
            const float Mt = sm.M[k], St = sm.S[k], Md = sm.M[g + 1 + k], Sd = sm.S[g + 1 + k];
            if (threadIdx.x == 0) sm.result = -1;
            for (int round = 0; round < MAX_TRIALS / NCW; ++round) {
                const uint32_t t = static_cast<uint32_t>(round * NCW + warp);
                const int x = race_p(P, trow, tp, Mt, key, t, static_cast<uint32_t>(k), lane);
                if (lane == 0) {
                    uint64_t w[4];
                    philox_group(w, key, STREAM_ACCEPT, t, static_cast<uint32_t>(k), 0);
                    const float v = uniform24(w[0]);
                    const float p = prob(P, tp, x, Mt, St);
                    const float q = prob(P, dp, x, Md, Sd);
                    sm.trial_x[warp] = x;
                    sm.trial_acc[warp] = (q <= (1.0f - v) * p) ? 1 : 0;
                }
                consumer_sync();
                if (threadIdx.x == 0) {
                    for (int w = 0; w < NCW; ++w)
                        if (sm.trial_acc[w]) {
                            sm.result = sm.trial_x[w];
                            break;
                        }
                }
                consumer_sync();
                if (sm.result >= 0) break;
            }
            const bool fallback = sm.result < 0;
            if (fallback || P.out_Z) {
                residual_pass(P, b, tp, dp, Mt, St, Md, Sd, sm, warp, lane);
                if (fallback) {
                    if (warp == 0) {
                        const int x = race_resid(P, b, tp, dp, Mt, St, Md, Sd, key, static_cast<uint32_t>(k), lane);
                        if (lane == 0) sm.result = x;
                    }
                    consumer_sync();
                }
            }
        }
        // 4. Outputs.
        const int res = sm.result;
        for (int i = threadIdx.x; i <= g; i += NCW * 32) {
            int v = -1;
            if (i < k) v = P.tokens[static_cast<size_t>(b) * g + i];
            else if (i == k) v = res;
            P.out_tokens[static_cast<size_t>(b) * (g + 1) + i] = v;
        }
        if (threadIdx.x == 0) {
            P.accept_count[b] = k;
            if (P.row_status) P.row_status[b] = 0;
            if (P.out_Z) P.out_Z[b] = (k == g) ? 1.0f : sm.Z;
            P.counter[b] = 0u;
        }
        consumer_sync();
    }
};

// =====================================================================================
// Greedy verify, T = 0
// =====================================================================================
struct GreedyParams {
    long long total_items;
    int nc, nb, V;
    unsigned *counter;
    unsigned *err;
    const unsigned char *target;
    const int32_t *tokens;
    int B, gamma, R;  // R = gamma + 1
    int32_t *accept_count, *out_tokens, *row_status;
    int2 *best;  // [B*R*nb] (max value bits, argmax id); id -2 marks a bad block
};

struct GreedySmem {
    int a[33];
    int bad;
};

template <int DT> struct GreedyOp {
    using Params = GreedyParams;
    using Smem = GreedySmem;
    static constexpr int EB = DType<DT>::BYTES;

    __device__ static __forceinline__ const void *row_ptr(const Params &P, long long row)
    {
        return P.target + static_cast<size_t>(row) * static_cast<size_t>(P.V) * EB;
    }
    __device__ static __forceinline__ int group(const Params &P, long long row) { return static_cast<int>(row / P.R); }
    __device__ static __forceinline__ int items_per_group(const Params &P) { return P.R * P.nc; }

    __device__ static __forceinline__ void block(const Params &P, long long row, int beta, float v[32], int, int lane)
    {
        float bv = -INFINITY;
        int bi = INT_MAX;
        bool nan = false;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            const float x = v[e];
            nan |= (x != x);
            if (x > bv) {  // strict: the first (lowest) id keeps a tie; -0.0 == +0.0
                bv = x;
                bi = lane_index<DT>(lane, e);
            }
        }
        warp_argmax(bv, bi);
        nan = __any_sync(0xffffffffu, nan);
        if (lane == 0) {
            int2 o;
            if (nan || bv == INFINITY) o = make_int2(0x7fc00000, -2);
            else o = make_int2(__float_as_int(bv), bi == INT_MAX ? INT_MAX : beta * G + bi);
            P.best[row * P.nb + beta] = o;
        }
    }

    __device__ static void finalize(const Params &P, int b, Smem &sm, int warp, int lane)
    {
        const int g = P.gamma, R = P.R;
        if (threadIdx.x == 0) sm.bad = 0;
        consumer_sync();
        for (int rho = warp; rho < R; rho += NCW) {
            const int2 *bb = P.best + (static_cast<long long>(b) * R + rho) * P.nb;
            float bv = -INFINITY;
            int bi = INT_MAX;
            bool bad = false;
            for (int beta = lane; beta < P.nb; beta += 32) {
                const int2 o = __ldcg(&bb[beta]);
                if (o.y == -2) {
                    bad = true;
                } else {
                    const float v = __int_as_float(o.x);
                    if (v > bv || (v == bv && o.y < bi)) {
                        bv = v;
                        bi = o.y;
                    }
                }
            }
            warp_argmax(bv, bi);
            bad = __any_sync(0xffffffffu, bad);
            if (lane == 0) {
                sm.a[rho] = bi;
                if (bad || bv == -INFINITY || bi == INT_MAX) atomicOr(&sm.bad, 1);
            }
        }
        if (warp == 0 && lane < g) {
            const int x = P.tokens[static_cast<size_t>(b) * g + lane];
            if (x < 0 || x >= P.V) atomicOr(&sm.bad, 1);
        }
        consumer_sync();
        if (warp == 0) {
            if (sm.bad) {
                for (int i = lane; i <= g; i += 32) P.out_tokens[static_cast<size_t>(b) * (g + 1) + i] = -1;
                if (lane == 0) {
                    P.accept_count[b] = -1;
                    if (P.row_status) P.row_status[b] = STATUS_BAD_ROW;
                }
            } else {
                int x = 0;
                bool acc = false;
                if (lane < g) {
                    x = P.tokens[static_cast<size_t>(b) * g + lane];
                    acc = (x == sm.a[lane]);
                }
                const unsigned mask = __ballot_sync(0xffffffffu, acc);
                const unsigned all = (g == 32) ? 0xffffffffu : ((1u << g) - 1u);
                const int k = ((mask & all) == all) ? g : (__ffs(~mask) - 1);
                for (int i = lane; i <= g; i += 32) {
                    int v = -1;
                    if (i < k) v = P.tokens[static_cast<size_t>(b) * g + i];
                    else if (i == k) v = sm.a[k];
                    P.out_tokens[static_cast<size_t>(b) * (g + 1) + i] = v;
                }
                if (lane == 0) {
                    P.accept_count[b] = k;
                    if (P.row_status) P.row_status[b] = 0;
                }
            }
            if (lane == 0) P.counter[b] = 0u;
        }
        consumer_sync();
    }
};

// =====================================================================================
// Host launch
// =====================================================================================
template <class Op, int DT> static cudaError_t launch_op(const typename Op::Params &P, bool tma, cudaStream_t st)
{
    void (*kern)(const typename Op::Params) = tma ? stream_kernel<Op, DT, true> : stream_kernel<Op, DT, false>;
    const int smem = tma ? stages<DT>() * CHUNK * DType<DT>::BYTES : 0;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, THREADS, smem)) != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const long long cap = static_cast<long long>(per_sm) * sms;
    const int grid = static_cast<int>(P.total_items < cap ? P.total_items : cap);
    kern<<<grid, THREADS, smem, st>>>(P);
    return cudaGetLastError();
}

size_t chain_ws_bytes(int B, int gamma, int V)
{
    const size_t nb = blocks_per_row(V), R = 2 * static_cast<size_t>(gamma) + 1;
    size_t n = WS_HEADER;
    n += align256(static_cast<size_t>(B) * 4);       // counters
    n += align256(static_cast<size_t>(B) * R * nb * 8); // block statistics
    n += align256(static_cast<size_t>(B) * nb * 4);  // residual block masses
    const size_t gr = greedy_ws_bytes(B, gamma, V);
    return n > gr ? n : gr;
}

size_t greedy_ws_bytes(int B, int gamma, int V)
{
    const size_t nb = blocks_per_row(V), R = static_cast<size_t>(gamma) + 1;
    return WS_HEADER + align256(static_cast<size_t>(B) * 4) + align256(static_cast<size_t>(B) * R * nb * 8);
}

cudaError_t launch_chain(const ChainLaunch &L, cudaStream_t st)
{
    ChainParams P{};
    P.V = L.V;
    P.nb = blocks_per_row(L.V);
    P.nc = chunks_per_row(L.V);
    P.B = L.B;
    P.gamma = L.gamma;
    P.R = 2 * L.gamma + 1;
    P.total_items = static_cast<long long>(L.B) * P.R * P.nc;
    unsigned char *ws = static_cast<unsigned char *>(L.ws);
    P.err = reinterpret_cast<unsigned *>(ws);
    size_t off = WS_HEADER;
    P.counter = reinterpret_cast<unsigned *>(ws + off);
    off += align256(static_cast<size_t>(L.B) * 4);
    P.stats = reinterpret_cast<float2 *>(ws + off);
    off += align256(static_cast<size_t>(L.B) * P.R * P.nb * 8);
    P.resid = reinterpret_cast<float *>(ws + off);
    P.target = static_cast<const unsigned char *>(L.target);
    P.draft = static_cast<const unsigned char *>(L.draft);
    P.tokens = L.tokens;
    P.r = L.r;
    P.keys = L.keys;
    P.invT = 1.0f / L.T;
    P.c2 = 1.4426950408889634f / L.T;
    P.accept_count = L.accept_count;
    P.out_tokens = L.out_tokens;
    P.out_pq = L.out_pq;
    P.out_Z = L.out_Z;
    P.row_status = L.row_status;
    return L.dtype == 0 ? launch_op<ChainOp<0>, 0>(P, L.tma, st) : launch_op<ChainOp<1>, 1>(P, L.tma, st);
}

cudaError_t launch_greedy(const ChainLaunch &L, cudaStream_t st)
{
    GreedyParams P{};
    P.V = L.V;
    P.nb = blocks_per_row(L.V);
    P.nc = chunks_per_row(L.V);
    P.B = L.B;
    P.gamma = L.gamma;
    P.R = L.gamma + 1;
    P.total_items = static_cast<long long>(L.B) * P.R * P.nc;
    unsigned char *ws = static_cast<unsigned char *>(L.ws);
    P.err = reinterpret_cast<unsigned *>(ws);
    size_t off = WS_HEADER;
    P.counter = reinterpret_cast<unsigned *>(ws + off);
    off += align256(static_cast<size_t>(L.B) * 4);
    P.best = reinterpret_cast<int2 *>(ws + off);
    P.target = static_cast<const unsigned char *>(L.target);
    P.tokens = L.tokens;
    P.accept_count = L.accept_count;
    P.out_tokens = L.out_tokens;
    P.row_status = L.row_status;
    return L.dtype == 0 ? launch_op<GreedyOp<0>, 0>(P, L.tma, st) : launch_op<GreedyOp<1>, 1>(P, L.tma, st);
}

}  // namespace spv
