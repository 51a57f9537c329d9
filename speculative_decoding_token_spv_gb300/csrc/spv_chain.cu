// spv_chain.cu -- chain verify (T > 0) and greedy verify (T = 0) kernels.
//
// Chain verify, "Speculative Decoding: How Draft-Model Parallelism Cuts LLM
// Inference Latency", section "The four-phase loop", steps 2-4:
//   one pass over the gamma+1 target rows and gamma draft rows of every
//   sequence computes, per 1024-logit sampler block, the block max m and
//   S = sum exp((z - m) / T).  The finalize grid (one CTA per sequence)
//   merges the blocks into row softmax statistics, runs the accept test
//   r_i q_i(x_i) <= p_i(x_i) for every draft token, finds the first
//   rejection with a warp ballot, and draws the emitted token: the bonus from
//   p_gamma, or the residual norm(max(0, p_k - q_k)) by rejection trials from
//   p_k (one trial per warp per round).  Draws use the three-level
//   exponential race (blocks from the per-block statistics, then sub-blocks
//   and ids inside a re-read 1024-logit block), so no row is read twice in
//   full from HBM.
//
// Greedy verify, "Speculative Pipeline Decoding", streaming verification
// (T = 0: a draft token stands only if it is the target argmax): the same
// pass over the target rows keeps per-block (max, lowest argmax id); the
// finalize CTA of a sequence compares each draft token with its row argmax.
//
// Both finalizers can also key the outcome (k, emitted token) against the
// sequence's speculation-cache entries ("Speculative Speculative Decoding",
// Algorithm 1 and Figure 2) and write the hit slot, and the chain finalizer
// verifies Saguaro-sampled drafts (cached candidates down-weighted by C).
//
// Tree verify (multi-round speculative sampling over a draft token tree per
// sequence, greedy descent at T = 0) reuses the streaming pass and the draws;
// see the tree section below.
#include "spv_internal.h"
#include "spv_stream.cuh"

#include <climits>

#include "spv.h"

static_assert(spv::CACHE_POSITIONS >= SPV_MAX_GAMMA + 1, "cache offsets must cover gamma + 1 positions");

namespace spv {

// =====================================================================================
// Chain verify, T > 0
// =====================================================================================
struct ChainParams {
    long long total_items;
    int nc, nb, V;
    unsigned *err;
    const unsigned char *target, *draft;
    const int32_t *tokens;
    const float *r;
    const uint64_t *keys;
    int B, gamma, R;
    int nt, nd;      // target / draft rows per sequence (chain: gamma + 1, gamma; tree: N, N)
    float invT, c2;  // 1/T and log2(e)/T
    int vec;         // rows 16-byte aligned: vector loads in finalize
    int32_t *accept_count, *out_tokens;
    float *out_pq, *out_Z;
    int32_t *row_status;
    float2 *stats;   // [B*R*nb] (block max of z, sum exp((z - max)/T)); NaN max = bad block
    float *resid;    // [B*nb] residual block masses (direct draw / normaliser only)
    CacheLookup cache;
    const int32_t *tree_parent;  // tree verify: [B, N] parents
    int32_t *tree_nodes;         // tree verify: [B, N] accepted nodes out (optional)
    int cs;                      // tree verify: finalize CTAs per sequence (one cluster)
    unsigned *tree_bar;          // tree verify: [B][2] barrier of a sequence's CTAs
    int sag;         // Saguaro sampling: the draft distribution at position i divides its
    float invC;      // cached candidates' (cache lists) probability by C (invC = 1/C)
};

constexpr int FW = 16;            // widest chain finalize CTA (warps; one residual trial each per round)
constexpr int STAT_CACHE = 4096;  // target-row block statistics staged in shared memory when they fit

struct ChainSmem {
    float2 st[STAT_CACHE];  // target rows: (block max, S_beta), or the race factor 2^((M - m) c2) / S_beta
                            // (-1 if empty) in place of S_beta when the merge staged factors (tree)
    float M[2 * 64 + 1];    // row max of the raw logits (chain: 2 gamma + 1 rows; tree: 2 N)
    float S[2 * 64 + 1];    // row sum exp((z - M)/T)
    int x[64];              // draft tokens (tree: node tokens)
    float rr[64];           // accept uniforms
    float zt[64], zd[64];   // target / draft logit of each draft token
    int bad;
    int k;
    int cached;
    int trial_x[2][FW];     // trial outcomes of a round (two buffers: rounds alternate)
    int trial_acc[2][FW];
    int result;
    int gflag;              // tree: outcome of the last barrier of the sequence's CTAs
    float Z;
    uint64_t key;
    int sag_id[32][64];  // Saguaro: cached candidates of draft position i (-1: none / repeated)
    int par[64];         // tree: parent of each node
};

// Barrier of the FWV warps of a chain finalize CTA.
template <int FWV> __device__ __forceinline__ void fin_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(FWV * 32) : "memory");
}

// Whether id x is among a Saguaro position's cached candidates (whole warp,
// same x).
__device__ __forceinline__ bool sag_member(const int *ids, int x, int lane)
{
    return __any_sync(0xffffffffu, ids[lane] == x || ids[32 + lane] == x);
}

// Residual mass max(0, p(x) - q(x)) from the logits of x: p and q are each
// rounded to fp32 before the difference (no fused multiply-add across them),
// so identical target and draft logits give exactly 0.
__device__ __forceinline__ float resid_mass(float zt, float zd, float Mt, float it, float Md, float id, float invT)
{
    const float p = __fmul_rn(expf((zt - Mt) * invT), it);
    const float q = __fmul_rn(expf((zd - Md) * invT), id);
    return fmaxf(__fsub_rn(p, q), 0.f);
}

// The same with the draft probability scaled by wq (Saguaro: 1/C on cached ids).
__device__ __forceinline__ float resid_mass_w(float zt, float zd, float Mt, float it, float Md, float id, float invT,
                                              float wq)
{
    const float p = __fmul_rn(expf((zt - Mt) * invT), it);
    const float q = __fmul_rn(__fmul_rn(expf((zd - Md) * invT), id), wq);
    return fmaxf(__fsub_rn(p, q), 0.f);
}

// Word j (0..3) of a Philox group without indexing the register array.
__device__ __forceinline__ uint32_t word_of(const uint32_t w[4], int j)
{
    return j == 0 ? w[0] : (j == 1 ? w[1] : (j == 2 ? w[2] : w[3]));
}

// The variates of one draw -- a residual trial, or the bonus (trial 0) --
// held by one warp.  Lane l holds the exponentials E = -ln U of blocks
// 4 (l + 32 h) + e (h < 2, e < 4: rows of up to PRE_BLOCKS blocks), of
// sub-block l of the winning block, of id offset l in the winning sub-block,
// and the trial's acceptance word.  None depends on the row, the position or
// the statistics, so a finalize computes the first round's before its
// dependent-grid wait.
constexpr int PRE_BLOCKS = 160;  // 40 Philox groups: every lane's first, lanes 0..7's second
struct DrawVariates {
    float eb[2][4];
    float es, ex;
    uint32_t aw;
};

// A warp's DrawVariates parked in shared memory, lane-major: the values of
// lane l at [i * 32 + l].  Computing a round's variates before the
// dependent-grid wait only helps if they stay computed: in registers the
// compiler may recompute them where they are used.
constexpr int DRAW_SLOT_FLOATS = 11 * 32;
__device__ __forceinline__ void store_draw(float *slot, const DrawVariates &dv, int lane)
{
#pragma unroll
    for (int i = 0; i < 8; ++i) slot[i * 32 + lane] = dv.eb[i >> 2][i & 3];
    slot[8 * 32 + lane] = dv.es;
    slot[9 * 32 + lane] = dv.ex;
    slot[10 * 32 + lane] = __uint_as_float(dv.aw);
}
__device__ __forceinline__ void load_draw(DrawVariates &dv, const float *slot, int lane)
{
#pragma unroll
    for (int i = 0; i < 8; ++i) dv.eb[i >> 2][i & 3] = slot[i * 32 + lane];
    dv.es = slot[8 * 32 + lane];
    dv.ex = slot[9 * 32 + lane];
    dv.aw = __float_as_uint(slot[10 * 32 + lane]);
}

// At most two Philox calls per lane: every lane its block group (lane), then
// lanes 0..7 block group lane + 32, lanes 8..15 sub-block group lane - 8,
// lanes 16..23 id group lane - 16, lane 24 the acceptance group; the
// sub-block, id and acceptance words then reach their lanes by shuffles.
__device__ __forceinline__ void draw_variates(DrawVariates &dv, uint64_t key, uint32_t trial, int nb, int lane)
{
    const bool pre = nb <= PRE_BLOCKS;
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    if (pre && 4 * lane < nb) philox_group(w, key, STREAM_BLOCK, trial, static_cast<uint32_t>(lane));
#pragma unroll
    for (int e = 0; e < 4; ++e) dv.eb[0][e] = expo(w[e]);
    uint32_t stream = STREAM_ACCEPT, grp = 0u;
    bool run = true;
    if (lane < 8) {
        stream = STREAM_BLOCK;
        grp = static_cast<uint32_t>(lane + 32);
        run = pre && 4 * (lane + 32) < nb;
    } else if (lane < 16) {
        stream = STREAM_SUB;
        grp = static_cast<uint32_t>(lane - 8);
    } else if (lane < 24) {
        stream = STREAM_TOKEN;
        grp = static_cast<uint32_t>(lane - 16);
    } else {
        run = lane == 24;
    }
    uint32_t v[4] = {0u, 0u, 0u, 0u};
    if (run) philox_group(v, key, stream, trial, grp);
#pragma unroll
    for (int e = 0; e < 4; ++e) dv.eb[1][e] = expo(v[e]);
    const int ss = 8 + (lane >> 2), st = 16 + (lane >> 2);  // lanes holding this lane's sub-block / id group
    uint32_t ws[4], wt[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        ws[e] = __shfl_sync(0xffffffffu, v[e], ss);
        wt[e] = __shfl_sync(0xffffffffu, v[e], st);
    }
    dv.es = expo(word_of(ws, lane & 3));
    dv.ex = expo(word_of(wt, lane & 3));
    dv.aw = __shfl_sync(0xffffffffu, v[0], 24);
}

template <int DT> struct ChainOp {
    using Params = ChainParams;
    using Smem = ChainSmem;
    static constexpr int EB = DType<DT>::BYTES;

    // Row rho of sequence b: target rows 0 .. nt-1, then draft rows.
    __device__ static __forceinline__ const unsigned char *row_of(const Params &P, int b, int rho)
    {
        if (rho < P.nt)
            return P.target + (static_cast<size_t>(b) * P.nt + rho) * static_cast<size_t>(P.V) * EB;
        return P.draft + (static_cast<size_t>(b) * P.nd + (rho - P.nt)) * static_cast<size_t>(P.V) * EB;
    }
    __device__ static __forceinline__ const void *row_ptr(const Params &P, long long row)
    {
        const int b = static_cast<int>(div_row(row, P.R));
        return row_of(P, b, static_cast<int>(row - static_cast<long long>(b) * P.R));
    }

    static constexpr int CTAS_PER_SM = DT == 0 ? 2 : 4;

    // From the staged block.  bf16 stays packed for the max (bf16x2 max,
    // NaN ignored like fmaxf) and is widened only for the exponentials.
    __device__ static __forceinline__ void block_smem(const Params &P, long long row, int beta,
                                                      const unsigned char *blk, int valid, int lane)
    {
        if (DT == 0) {
            float v[32];
            load_block_smem<DT>(v, blk, lane);
            mask_tail<DT>(v, valid, lane);
            block(P, row, beta, v, valid, lane);
            return;
        }
        uint32_t w[16];
        const uint4 *p = reinterpret_cast<const uint4 *>(blk);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 t = p[j * 32 + lane];
            w[4 * j] = t.x;
            w[4 * j + 1] = t.y;
            w[4 * j + 2] = t.z;
            w[4 * j + 3] = t.w;
        }
        if (valid < G) {  // element 2h / 2h+1 of word h of vector j: j*256 + lane*8 + 2h (+1)
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const int e0 = (q >> 2) * 256 + lane * 8 + 2 * (q & 3);
                if (e0 >= valid) w[q] = (w[q] & 0xffff0000u) | 0xff80u;       // -inf in the low half
                if (e0 + 1 >= valid) w[q] = (w[q] & 0x0000ffffu) | 0xff800000u; // and the high half
            }
        }
        __nv_bfloat162 mx[8];
#pragma unroll
        for (int a = 0; a < 8; ++a)
            mx[a] = __hmax2(*reinterpret_cast<const __nv_bfloat162 *>(&w[a]),
                            *reinterpret_cast<const __nv_bfloat162 *>(&w[a + 8]));
#pragma unroll
        for (int a = 0; a < 4; ++a) mx[a] = __hmax2(mx[a], mx[a + 4]);
        mx[0] = __hmax2(__hmax2(mx[0], mx[1]), __hmax2(mx[2], mx[3]));
        const float m = warp_max_redux(fmaxf(__low2float(mx[0]), __high2float(mx[0])));
        const float mu = (m == -INFINITY) ? 0.f : m;
        const float mc = mu * P.c2;
        const float delta = fmaf(mu, P.c2, -mc);
        // z c2 - mc and the running sums on packed pairs (elements 2h, 2h + 1 of a word)
        const unsigned long long c2x2 = pack2(P.c2, P.c2), nmc2 = pack2(-mc, -mc);
        unsigned long long acc[2] = {0ull, 0ull};
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            float a0, a1;
            unpack2(ffma2(pack2(__uint_as_float(w[q] << 16), __uint_as_float(w[q] & 0xffff0000u)), c2x2, nmc2), a0, a1);
            acc[q & 1] = fadd2(acc[q & 1], pack2(fast_exp2(a0), fast_exp2(a1)));
        }
        float sa[4];
        unpack2(acc[0], sa[0], sa[1]);
        unpack2(acc[1], sa[2], sa[3]);
        float s = (sa[0] + sa[1]) + (sa[2] + sa[3]);
        s = warp_sum(s);
        if (lane == 0) {
            s = fmaf(-s * 0.6931471805599453f, delta, s);
            P.stats[row * P.nb + beta] = isnan(s) ? make_float2(__int_as_float(0x7fffffff), 0.f) : make_float2(m, s);
        }
    }

    // Block statistics: m = max z (raw), s = sum exp((z - m) / T).
    // The max is a tree of three-input maxima and one warp redux (NaN
    // ignored, like fmaxf: a NaN shows up in the sum); the sum runs as 4
    // independent chains; each term is
    // ex2(z * c2 - mc) with mc = m * c2 rounded, one FFMA, and the rounding
    // of mc (delta = m * c2 - mc, exact by FMA) is removed from the sum once:
    // sum ex2((z - m) c2) = 2^-delta * sum ex2(z c2 - mc).
    __device__ static __forceinline__ void block(const Params &P, long long row, int beta, float v[32], int, int lane)
    {
        float t[10];
#pragma unroll
        for (int a = 0; a < 10; ++a) t[a] = fmax3(v[3 * a], v[3 * a + 1], v[3 * a + 2]);
        const float u = fmax3(fmax3(t[0], t[1], t[2]), fmax3(t[3], t[4], t[5]), fmax3(t[6], t[7], t[8]));
        const float m = warp_max_redux(fmax3(u, t[9], fmaxf(v[30], v[31])));
        const float mu = (m == -INFINITY) ? 0.f : m;
        const float mc = mu * P.c2;
        const float delta = fmaf(mu, P.c2, -mc);
        const unsigned long long c2x2 = pack2(P.c2, P.c2), nmc2 = pack2(-mc, -mc);
        unsigned long long acc[2] = {0ull, 0ull};
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
            float a0, a1;
            unpack2(ffma2(pack2(v[e], v[e + 1]), c2x2, nmc2), a0, a1);
            acc[(e >> 1) & 1] = fadd2(acc[(e >> 1) & 1], pack2(fast_exp2(a0), fast_exp2(a1)));
        }
        float sa[4];
        unpack2(acc[0], sa[0], sa[1]);
        unpack2(acc[1], sa[2], sa[3]);
        float s = (sa[0] + sa[1]) + (sa[2] + sa[3]);
        s = warp_sum(s);
        if (lane == 0) {
            s = fmaf(-s * 0.6931471805599453f, delta, s);  // s * 2^-delta, |delta| < 1e-5
            // NaN anywhere, or +inf (then inf - inf), makes s NaN.
            P.stats[row * P.nb + beta] = isnan(s) ? make_float2(__int_as_float(0x7fffffff), 0.f) : make_float2(m, s);
        }
    }

    __device__ static __forceinline__ float prob(const Params &P, const unsigned char *rowp, int x, float M, float S)
    {
        return expf((DType<DT>::load(rowp, x) - M) * P.invT) / S;
    }

    // Level 1 of a draw from softmax(row rho / T): the block with the
    // smallest E_beta / W_beta, W_beta = 2^((m_beta - M) c2) S_beta up to the
    // row normaliser, i.e. arrival E_beta * f_beta with the factor
    // f_beta = 2^((M - m_beta) c2) / S_beta, staged by the merge when
    // `staged` (else computed here from the block statistics, in shared
    // memory when they fit).  The exponentials E_beta come from dv when it
    // holds them (rows of up to PRE_BLOCKS blocks), else from Philox here.
    // Every lane gets the winner.
    __device__ static int race_blocks_p(const Params &P, const Smem &sm, int b, int rho, float M, uint64_t key,
                                        uint32_t trial, int lane, const DrawVariates &dv, bool staged)
    {
        float best = INFINITY;
        int bi = INT_MAX;
        auto visit = [&](int g, const float E[4]) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int beta = 4 * g + e;
                float f;
                if (beta >= P.nb) {
                    f = -1.f;
                } else if (sm.cached) {
                    const float2 st = sm.st[rho * P.nb + beta];
                    f = staged ? st.y : (st.y > 0.f ? __fdividef(fast_exp2((M - st.x) * P.c2), st.y) : -1.f);
                } else {
                    const float2 st = __ldcg(&P.stats[(static_cast<long long>(b) * P.R + rho) * P.nb + beta]);
                    f = st.y > 0.f ? fast_exp2((M - st.x) * P.c2) / st.y : -1.f;
                }
                if (f >= 0.f) {
                    const float A = arrival(E[e], f);
                    if (A < best) {
                        best = A;
                        bi = beta;
                    }
                }
            }
        };
        if (P.nb <= PRE_BLOCKS && sm.cached && !staged) {
            // the lane's eight blocks 4 lane + 128 h + e as independent
            // arrivals (loads, exponentials and divisions all in flight),
            // then a pairwise minimum in index order (ties to the lower one)
            float A[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int beta = 4 * lane + 128 * (j >> 2) + (j & 3);
                A[j] = INFINITY;
                if (beta < P.nb) {
                    const float2 st = sm.st[rho * P.nb + beta];
                    if (st.y > 0.f) A[j] = arrival(dv.eb[j >> 2][j & 3], __fdividef(fast_exp2((M - st.x) * P.c2), st.y));
                }
            }
            int I[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) I[j] = 4 * lane + 128 * (j >> 2) + (j & 3);
#pragma unroll
            for (int w = 1; w < 8; w *= 2)
#pragma unroll
                for (int j = 0; j + w < 8; j += 2 * w)
                    if (A[j + w] < A[j]) {
                        A[j] = A[j + w];
                        I[j] = I[j + w];
                    }
            best = A[0];
            bi = best == INFINITY ? INT_MAX : I[0];
        } else if (P.nb <= PRE_BLOCKS) {
            if (4 * lane < P.nb) visit(lane, dv.eb[0]);
            if (4 * (lane + 32) < P.nb) visit(lane + 32, dv.eb[1]);
        } else {
            for (int g = lane; 4 * g < P.nb; g += 32) {
                uint32_t w[4];
                philox_group(w, key, STREAM_BLOCK, trial, static_cast<uint32_t>(g));
                const float E[4] = {expo(w[0]), expo(w[1]), expo(w[2]), expo(w[3])};
                visit(g, E);
            }
        }
        warp_argmin(best, bi);
        return bi;
    }

    // Max of the raw logits of block beta of target row rho.
    __device__ static __forceinline__ float block_max(const Params &P, const Smem &sm, int b, int rho, int beta)
    {
        return sm.cached ? sm.st[rho * P.nb + beta].x
                         : __ldcg(&P.stats[(static_cast<long long>(b) * P.R + rho) * P.nb + beta]).x;
    }

    // Block beta of a row into a warp's buffer of G floats (-inf past V):
    // 16-byte vector loads when the rows are aligned, all in flight at once.
    __device__ static __forceinline__ void load_block(const Params &P, const unsigned char *rowp, int beta, float *buf,
                                                      int lane)
    {
        const int base = beta * G;
        if (P.vec) {
#pragma unroll
            for (int j = 0; j < G / 128; ++j) {
                const int i = 4 * (lane + 32 * j);
                float f[4];
                if (base + i < P.V) {
                    if (DT == 0) {
                        const float4 t = __ldg(reinterpret_cast<const float4 *>(rowp) + ((base + i) >> 2));
                        f[0] = t.x; f[1] = t.y; f[2] = t.z; f[3] = t.w;
                    } else {
                        const uint2 t = __ldg(reinterpret_cast<const uint2 *>(rowp) + ((base + i) >> 2));
                        f[0] = __uint_as_float(t.x << 16); f[1] = __uint_as_float(t.x & 0xffff0000u);
                        f[2] = __uint_as_float(t.y << 16); f[3] = __uint_as_float(t.y & 0xffff0000u);
                    }
                } else {
                    f[0] = f[1] = f[2] = f[3] = -INFINITY;
                }
                *reinterpret_cast<float4 *>(buf + i) = make_float4(f[0], f[1], f[2], f[3]);
            }
        } else {
#pragma unroll 8
            for (int j = 0; j < G / 32; ++j) {
                const int i = lane + 32 * j;
                buf[i] = base + i < P.V ? DType<DT>::load(rowp, base + i) : -INFINITY;
            }
        }
        __syncwarp();
    }

    // Levels 2 and 3 of a draw from softmax(row / T) inside block beta (block
    // max mb) whose logits are in buf: lane l owns sub-block l (ids
    // base + 32 l + i) for the sub-block race, then id base + 32 s* + l for
    // the id race, with the exponentials of dv (sub-block l, id offset l).
    __device__ static int race_in_block_p(const Params &P, const float *buf, int beta, float mb,
                                          const DrawVariates &dv, int lane)
    {
        const int base = beta * G;
        // sub-block mass relative to the block max (skewed reads: no bank
        // conflicts), four partial sums in flight
        float w4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
        for (int i = 0; i < SUB; ++i)
            w4[i & 3] += fast_exp2((buf[SUB * lane + ((i + lane) & (SUB - 1))] - mb) * P.c2);
        const float ws = (w4[0] + w4[1]) + (w4[2] + w4[3]);
        float A = ws > 0.f ? arrival(dv.es, 1.f / ws) : INFINITY;
        int si = lane;
        warp_argmin(A, si);
        const int x = base + SUB * si + lane;
        const float z = buf[SUB * si + lane];
        const float msw = warp_max_redux(z);  // max of the winning sub-block
        float Ax = (x < P.V && z != -INFINITY) ? arrival(dv.ex, fast_exp2((msw - z) * P.c2)) : INFINITY;
        int xi = x;
        warp_argmin(Ax, xi);
        return xi;
    }

    // Row statistics of sequence b from its block statistics: one half-warp
    // per row, all rows at once, up to 16 loads per lane in flight together:
    // sm.M / sm.S = row max / sum exp((z - max) / T).  Target rows rho <
    // ncache keep (m_beta, S_beta) in sm.st for the draws (when they fit);
    // with FACTORS their race factors replace S_beta there (else the draws
    // compute the factors from (m_beta, S_beta) themselves).  A bad
    // row (NaN / +inf, no finite logit) gets S = NaN; with flag_all it also
    // sets sm.bad.  FWV warps.
    template <int FWV, bool FACTORS>
    __device__ static void merge_stats(const Params &P, int b, Smem &sm, int ncache, bool flag_all, int warp, int lane)
    {
        const int R = P.R, nb = P.nb;
        const int half = lane >> 4, hl = lane & 15;
        for (int rho0 = 0; rho0 < R; rho0 += 2 * FWV) {
            const int rho = rho0 + 2 * warp + half;
            const bool active = rho < R;
            const float2 *st = P.stats + (static_cast<long long>(b) * R + (active ? rho : 0)) * nb;
            const bool keep = active && rho < ncache && sm.cached;
            float m = -INFINITY, s = 0.f;
            bool bad = false;
            for (int base = 0; base < nb; base += 16 * 16) {
                float2 v[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int beta = base + 16 * u + hl;
                    v[u] = (active && beta < nb) ? __ldcg(&st[beta]) : make_float2(-INFINITY, 0.f);
                }
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int beta = base + 16 * u + hl;
                    bad |= isnan(v[u].x);
                    if (keep && beta < nb) sm.st[rho * nb + beta] = v[u];
                }
                // the max as a tree of three-input maxima (NaN ignored, like
                // fmaxf), the sum as four partial sums: short dependent chains
                float t6[6];
#pragma unroll
                for (int j = 0; j < 5; ++j) t6[j] = fmax3(v[3 * j].x, v[3 * j + 1].x, v[3 * j + 2].x);
                t6[5] = fmaxf(v[15].x, m);
                const float nm = fmax3(fmax3(t6[0], t6[1], t6[2]), fmax3(t6[3], t6[4], t6[5]), -INFINITY);
                if (nm != -INFINITY) {
                    // ex2.approx of arguments <= 0 (relative error ~2e-7 for the
                    // blocks near the row max, which carry the sum)
                    float acc[4] = {s > 0.f ? s * fast_exp2((m - nm) * P.c2) : 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int u = 0; u < 16; ++u)
                        if (v[u].y > 0.f) acc[u & 3] = fmaf(v[u].y, fast_exp2((v[u].x - nm) * P.c2), acc[u & 3]);
                    s = (acc[0] + acc[1]) + (acc[2] + acc[3]);
                    m = nm;
                }
            }
            float mw = m;
#pragma unroll
            for (int o = 8; o; o >>= 1) mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, o));
            s = (s > 0.f) ? s * fast_exp2((m - mw) * P.c2) : 0.f;
#pragma unroll
            for (int o = 8; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            const unsigned badm = __ballot_sync(0xffffffffu, bad);
            const bool rowbad = ((badm >> (16 * half)) & 0xffffu) != 0 || !(s > 0.f);
            if (active && hl == 0) {
                sm.M[rho] = mw;
                sm.S[rho] = rowbad ? __int_as_float(0x7fffffff) : s;
                if (rowbad && flag_all) atomicOr(&sm.bad, 1);
            }
            if (FACTORS && keep && !rowbad && mw != -INFINITY) {
                // entry beta was staged by this lane (beta = hl mod 16): no warp barrier needed
                for (int beta = hl; beta < nb; beta += 16) {
                    const float2 v = sm.st[rho * nb + beta];
                    sm.st[rho * nb + beta].y = v.y > 0.f ? fast_exp2((mw - v.x) * P.c2) / v.y : -1.f;
                }
            }
        }
    }

    // Direct race over the residual w = max(0, p - q) (after the rejection
    // trials all failed): block masses from residual_pass, then sub-blocks
    // and ids of the winning block (target and draft logits in tb / db).
    __device__ static int race_resid(const Params &P, int b, const unsigned char *tp, const unsigned char *dp, float Mt,
                                     float St, float Md, float Sd, uint64_t key, float *tb, float *db,
                                     const int *sids, float qs, int lane, const float *rb = nullptr)
    {
        if (!rb) rb = P.resid + static_cast<size_t>(b) * P.nb;  // the block masses of the residual
        float best = INFINITY;
        int bi = INT_MAX;
        for (int g = lane; 4 * g < P.nb; g += 32) {
            float W[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int beta = 4 * g + e;
                W[e] = beta < P.nb ? __ldcg(&rb[beta]) : 0.f;
            }
            uint32_t w[4];
            philox_group(w, key, STREAM_FB_BLOCK, 0, static_cast<uint32_t>(g));
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (W[e] > 0.f) {
                    const float A = arrival(expo(w[e]), 1.f / W[e]);
                    if (A < best) {
                        best = A;
                        bi = 4 * g + e;
                    }
                }
            }
        }
        warp_argmin(best, bi);
        if (bi == INT_MAX) return -1;  // no block with positive residual mass
        load_block(P, tp, bi, tb, lane);
        load_block(P, dp, bi, db, lane);
        const float it = 1.f / St, id = 1.f / Sd;
        const int base = bi * G;
        // Saguaro: bit e of lane l marks a cached id at base + 32 l + e (its q is scaled by 1/C)
        uint32_t smask = 0u;
        if (sids) {
            for (int j = 0; j < 64; ++j) {
                const int x = sids[j] - base;
                if (x >= 0 && x < G && (x >> 5) == lane) smask |= 1u << (x & 31);
            }
        }
        float ws = 0.f;
        for (int i = 0; i < SUB; ++i) {
            const int e = (i + lane) & (SUB - 1), o = SUB * lane + e;
            ws += resid_mass_w(tb[o], db[o], Mt, it, Md, id, P.invT, ((smask >> e) & 1u) ? P.invC * qs : qs);
        }
        uint32_t w[4];
        philox_group(w, key, STREAM_FB_SUB, 0, static_cast<uint32_t>(lane) >> 2);  // sub-block lane of the block
        float A = ws > 0.f ? arrival(expo(word_of(w, lane & 3)), 1.f / ws) : INFINITY;
        int si = lane;
        warp_argmin(A, si);
        const int x = base + SUB * si + lane;
        const int o = SUB * si + lane;
        const uint32_t wmask = __shfl_sync(0xffffffffu, smask, si);
        const float wx =
            x < P.V ? resid_mass_w(tb[o], db[o], Mt, it, Md, id, P.invT, ((wmask >> lane) & 1u) ? P.invC * qs : qs)
                    : 0.f;
        philox_group(w, key, STREAM_FB_TOKEN, 0, static_cast<uint32_t>(lane) >> 2);  // id offset lane of the sub-block
        float Ax = wx > 0.f ? arrival(expo(word_of(w, lane & 3)), 1.f / wx) : INFINITY;
        int xi = x;
        warp_argmin(Ax, xi);
        return xi;
    }

};

// The chain finalize at a given width: FWV warps, FWV residual trials per
// round.  Wider CTAs draw in fewer rounds; narrower ones fit two per SM.
template <int DT, int FWV, bool PRE = (FWV >= 16)> struct ChainFin : ChainOp<DT> {
    using Base = ChainOp<DT>;
    using Params = ChainParams;
    using Smem = ChainSmem;
    using Base::row_of;
    using Base::race_blocks_p;
    using Base::load_block;
    using Base::race_in_block_p;
    using Base::race_resid;
    using Base::block_max;

    // Residual masses w = max(0, p - q) of one row pair, per block, into
    // P.resid; returns Z = sum w in sm.Z.  All consumer warps.
    __device__ static void residual_pass(const Params &P, int b, const unsigned char *tp, const unsigned char *dp,
                                         float Mt, float St, float Md, float Sd, Smem &sm, int warp, int lane, float *tb,
                                         int k, float qs = 1.f)
    {
        const float it = 1.f / St, id = 1.f / Sd;
        for (int beta = warp; beta < P.nb; beta += FWV) {
            float part = 0.f;
            const int hi = min(P.V, (beta + 1) * G);
            for (int x = beta * G + lane; x < hi; x += 32)
                part += resid_mass_w(DType<DT>::load(tp, x), DType<DT>::load(dp, x), Mt, it, Md, id, P.invT, qs);
            part = warp_sum(part);
            if (lane == 0) P.resid[static_cast<size_t>(b) * P.nb + beta] = part;
        }
        fin_sync<FWV>();
        if (warp == 0) {
            float *rb = P.resid + static_cast<size_t>(b) * P.nb;
            if (P.sag) {
                // Saguaro: the cached ids' q is scaled by 1/C; correct their
                // blocks' masses in a shared copy (in list order: deterministic).
                for (int beta = lane; beta < P.nb; beta += 32) tb[beta] = __ldcg(&rb[beta]);
                float dlt[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int x = sm.sag_id[k][32 * h + lane];
                    dlt[h] = 0.f;
                    if (x >= 0) {
                        const float zt = DType<DT>::load(tp, x), zd = DType<DT>::load(dp, x);
                        dlt[h] = resid_mass_w(zt, zd, Mt, it, Md, id, P.invT, P.invC) -
                                 resid_mass(zt, zd, Mt, it, Md, id, P.invT);
                    }
                }
                __syncwarp();
                for (int j = 0; j < 64; ++j) {
                    const float dj = __shfl_sync(0xffffffffu, dlt[j >> 5], j & 31);
                    const int x = sm.sag_id[k][j];
                    if (lane == 0 && x >= 0) tb[x / G] += dj;
                }
                __syncwarp();
                float z = 0.f;
                for (int beta = lane; beta < P.nb; beta += 32) {
                    rb[beta] = tb[beta];
                    z += tb[beta];
                }
                z = warp_sum(z);
                if (lane == 0) sm.Z = z;
            } else {
                float z = 0.f;
                for (int beta = lane; beta < P.nb; beta += 32) z += __ldcg(&rb[beta]);
                z = warp_sum(z);
                if (lane == 0) sm.Z = z;
            }
        }
        fin_sync<FWV>();
    }

    static constexpr int FIN_WARPS = FWV;
    static constexpr bool PRE_DRAW = PRE;  // first round's variates drawn before the wait
    // per warp: one target and one draft block (and its parked variates)
    static constexpr int FIN_BUF_FLOATS = 2 * FWV * G + (PRE_DRAW ? FWV * DRAW_SLOT_FLOATS : 0);

    // Outputs of a bad row: -1 ids and count, NaN p / q / Z, status (bad row,
    // or timeout when a bounded wait of the streaming pass gave up), cache miss.
    __device__ static void write_bad_row(const Params &P, int b, int warp, int lane, int status = STATUS_BAD_ROW)
    {
        constexpr int NT = FWV * 32;
        const int g = P.gamma;
        for (int i = threadIdx.x; i <= g; i += NT) P.out_tokens[static_cast<size_t>(b) * (g + 1) + i] = -1;
        if (P.out_pq)
            for (int i = threadIdx.x; i < 2 * g; i += NT)
                P.out_pq[static_cast<size_t>(b) * 2 * g + i] = __int_as_float(0x7fffffff);
        if (threadIdx.x == 0) {
            P.accept_count[b] = -1;
            if (P.row_status) P.row_status[b] = status;
            if (P.out_Z) P.out_Z[b] = __int_as_float(0x7fffffff);
        }
        if (warp == 0) cache_lookup(P.cache, b, -1, -1, lane);
    }

    __device__ static void finalize(const Params &P, int b, Smem &sm, float *buf, int warp, int lane)
    {
        const int g = P.gamma, nb = P.nb;
        constexpr int NT = FWV * 32;
        float *tb = buf + warp * 2 * G, *db = tb + G;  // this warp's block buffers
        // A. Inputs that do not depend on the streaming grid: tokens, r, key
        //    and the logits of each draft token (overlaps the grid's tail).
        if (threadIdx.x == 0) {
            sm.bad = 0;
            sm.key = P.keys[b];
            sm.cached = ((g + 1) * nb <= STAT_CACHE) ? 1 : 0;
        }
        if (warp == 0 && lane < g) {
            const int x = P.tokens[static_cast<size_t>(b) * g + lane];
            sm.x[lane] = x;
            sm.rr[lane] = P.r[static_cast<size_t>(b) * g + lane];
            if (x >= 0 && x < P.V) {
                sm.zt[lane] = DType<DT>::load(row_of(P, b, lane), x);
                sm.zd[lane] = DType<DT>::load(row_of(P, b, g + 1 + lane), x);
            } else {
                sm.zt[lane] = sm.zd[lane] = 0.f;
            }
        }
        if (warp == 1) cache_prefetch(P.cache, b, lane);
        // Saguaro: each warp stages the cached ids of its draft positions
        // (repeats and ids outside [0, V) dropped) and their draft logits.
        constexpr int SAG_PER_WARP = (32 + FWV - 1) / FWV;
        float sz[SAG_PER_WARP][2];
        if (P.sag) {
#pragma unroll
            for (int u = 0; u < SAG_PER_WARP; ++u) {
                const int i = warp + u * FWV;
                sz[u][0] = sz[u][1] = 0.f;
                if (i < g) {
                    const int o0 = P.cache.off[i], F = P.cache.off[i + 1] - o0;
                    const int32_t *ids = P.cache.ids + static_cast<size_t>(b) * P.cache.n + o0;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int j = 32 * h + lane;
                        int x = j < F ? ids[j] : -1;
                        if (x < 0 || x >= P.V) x = -1;
                        sm.sag_id[i][j] = x;
                    }
                    __syncwarp();
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int j = 32 * h + lane;
                        const int x = sm.sag_id[i][j];
                        bool rep = false;
                        for (int j2 = 0; j2 < j && x >= 0; ++j2) rep |= sm.sag_id[i][j2] == x;
                        if (x >= 0 && !rep) sz[u][h] = DType<DT>::load(row_of(P, b, g + 1 + i), x);
                        else sz[u][h] = -INFINITY;
                    }
                    __syncwarp();
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        if (sz[u][h] == -INFINITY) sm.sag_id[i][32 * h + lane] = -1;
                    __syncwarp();
                }
            }
        }
        // The variates of the first round of residual trials (trial = warp;
        // warp 0's are also the bonus draw's) depend on inputs only: a CTA
        // with PRE_DRAW draws them while the streaming grid drains and parks
        // them in shared memory (the CTA that runs two per SM has no room: it
        // draws them where they are used).
        float *slot = buf + 2 * FWV * G + warp * DRAW_SLOT_FLOATS;
        if constexpr (PRE_DRAW) {
            DrawVariates dv;
            draw_variates(dv, __ldg(&P.keys[b]), static_cast<uint32_t>(warp), nb, lane);
            store_draw(slot, dv, lane);
        }
        asm volatile("griddepcontrol.wait;" ::: "memory");
        fin_sync<FWV>();
        if (warp == 0 && lane < g && (sm.x[lane] < 0 || sm.x[lane] >= P.V)) atomicOr(&sm.bad, 1);
        if (threadIdx.x == 32 && workspace_timed_out(P.err)) atomicOr(&sm.bad, 2);  // statistics incomplete
        // B. Row statistics from the block statistics (all rows at once).
        Base::template merge_stats<FWV, false>(P, b, sm, g + 1, true, warp, lane);
        fin_sync<FWV>();
        if (sm.bad) {
            write_bad_row(P, b, warp, lane, (sm.bad & 2) ? STATUS_TIMEOUT : STATUS_BAD_ROW);
            return;
        }
        if (P.sag) {
            // Saguaro: q_C's normaliser S - (1 - 1/C) * sum over the cached ids (at least S / C)
#pragma unroll
            for (int u = 0; u < SAG_PER_WARP; ++u) {
                const int i = warp + u * FWV;
                if (i < g) {
                    const float Md = sm.M[g + 1 + i], Sd = sm.S[g + 1 + i];
                    float c = 0.f;
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        if (sz[u][h] != -INFINITY) c += expf((sz[u][h] - Md) * P.invT);
                    c = warp_sum(c);
                    if (lane == 0) sm.S[g + 1 + i] = fmaxf(Sd - (1.f - P.invC) * c, Sd * P.invC);
                }
            }
            fin_sync<FWV>();
        }
        // C. Accept tests for every draft position and the first rejection by
        //    ballot, in every warp (the same values from shared memory give
        //    every warp the same k: no barrier between the tests and the
        //    draws); warp 0 writes p and q.
        int k;
        {
            bool acc = false;
            if (lane < g) {
                const float p = expf((sm.zt[lane] - sm.M[lane]) * P.invT) / sm.S[lane];
                float q = expf((sm.zd[lane] - sm.M[g + 1 + lane]) * P.invT) / sm.S[g + 1 + lane];
                if (P.sag) {
                    bool in = false;
                    for (int j = 0; j < 64; ++j) in |= sm.sag_id[lane][j] == sm.x[lane];
                    if (in) q = __fmul_rn(q, P.invC);
                }
                acc = (p > 0.f) && (sm.rr[lane] * q <= p);
                if (warp == 0 && P.out_pq) {
                    P.out_pq[(static_cast<size_t>(b) * g + lane) * 2] = p;
                    P.out_pq[(static_cast<size_t>(b) * g + lane) * 2 + 1] = q;
                }
            }
            const unsigned mask = __ballot_sync(0xffffffffu, acc);
            const unsigned all = (g == 32) ? 0xffffffffu : ((1u << g) - 1u);
            k = ((mask & all) == all) ? g : (__ffs(~mask) - 1);
        }
        const uint64_t key = sm.key;
        const unsigned char *tp = row_of(P, b, k);
        const float Mt = sm.M[k], St = sm.S[k];
        int res = -1;
        // D. The emitted token.
        if (k == g) {
            // Bonus: one draw from p_gamma (warp 0).
            if (warp == 0) {
                DrawVariates dv0;
                if constexpr (PRE_DRAW) load_draw(dv0, slot, lane);
                else draw_variates(dv0, key, 0u, nb, lane);
                const int beta = race_blocks_p(P, sm, b, k, Mt, key, 0u, lane, dv0, false);
                load_block(P, tp, beta, tb, lane);
                const int x = race_in_block_p(P, tb, beta, block_max(P, sm, b, k, beta), dv0, lane);
                if (lane == 0) sm.result = x;
            }
            fin_sync<FWV>();
            res = sm.result;
        } else {
            // Residual: rejection trials from p_k, FWV at a time (one per warp);
            // every thread reads the round's outcomes after one barrier (the
            // rounds alternate between two buffers, so the next round's
            // writes cannot meet a slower warp's reads).
            const unsigned char *dp = row_of(P, b, g + 1 + k);
            const float Md = sm.M[g + 1 + k], Sd = sm.S[g + 1 + k];
            for (int round = 0; round < MAX_TRIALS / FWV; ++round) {
                const uint32_t t = static_cast<uint32_t>(round * FWV + warp);
                const int buf2 = round & 1;
                DrawVariates dv;
                if (PRE_DRAW && round == 0) load_draw(dv, slot, lane);
                else draw_variates(dv, key, t, nb, lane);
                const int beta = race_blocks_p(P, sm, b, k, Mt, key, t, lane, dv, false);
                load_block(P, tp, beta, tb, lane);
                load_block(P, dp, beta, db, lane);
                const int x = race_in_block_p(P, tb, beta, block_max(P, sm, b, k, beta), dv, lane);
                const float wq = (P.sag && sag_member(sm.sag_id[k], x, lane)) ? P.invC : 1.f;
                if (lane == 0) {
                    const float v = uniform24(dv.aw);
                    const float p = expf((tb[x - beta * G] - Mt) * P.invT) / St;
                    const float q = __fmul_rn(expf((db[x - beta * G] - Md) * P.invT) / Sd, wq);
                    sm.trial_x[buf2][warp] = x;
                    sm.trial_acc[buf2][warp] = (q <= (1.0f - v) * p) ? 1 : 0;
                }
                fin_sync<FWV>();
                for (int w = 0; w < FWV; ++w)
                    if (sm.trial_acc[buf2][w]) {
                        res = sm.trial_x[buf2][w];
                        break;
                    }
                if (res >= 0) break;
            }
            const bool fallback = res < 0;
            if (fallback || P.out_Z) {
                residual_pass(P, b, tp, dp, Mt, St, Md, Sd, sm, warp, lane, tb, k);
                if (fallback) {
                    if (warp == 0) {
                        const int x = race_resid(P, b, tp, dp, Mt, St, Md, Sd, key, tb, db,
                                                 P.sag ? sm.sag_id[k] : nullptr, 1.f, lane);
                        if (lane == 0) sm.result = x;
                    }
                    fin_sync<FWV>();
                    res = sm.result;
                }
            }
        }
        // E. Outputs.  No residual mass at all (a draft token outside q's
        //    support with p = q elsewhere) leaves nothing to draw: bad row.
        if (res < 0) {
            write_bad_row(P, b, warp, lane);
            return;
        }
        for (int i = threadIdx.x; i <= g; i += NT) {
            int v = -1;
            if (i < k) v = sm.x[i];
            else if (i == k) v = res;
            P.out_tokens[static_cast<size_t>(b) * (g + 1) + i] = v;
        }
        if (threadIdx.x == 0) {
            P.accept_count[b] = k;
            if (P.row_status) P.row_status[b] = 0;
            if (P.out_Z) P.out_Z[b] = (k == g) ? 1.0f : sm.Z;
        }
        if (warp == FWV - 1) cache_lookup(P.cache, b, k, res, lane);
    }
};

// =====================================================================================
// Tree verify, T > 0 (multi-round speculative sampling over a token tree)
// =====================================================================================
// Rows per sequence: target rows 0..N-1 (p at node v), draft rows N..2N-1 (q
// at node v, from which v's children were drawn).  The finalize walks the
// tree from the root: the children c of node u are tested in index order
// against P_m = max(0, p_u - s_m q_u) / N_m (s_0 = 0, N_0 = 1, s_{m+1} = s_m +
// N_m, N_m = sum max(0, p_u - s_m q_u): a residual pass split over the
// sequence's cluster of finalize CTAs); the first accepted child is
// descended into; when all are rejected one token is drawn from P_m
// (rejection trials from p_u with q scaled by s_m, then the direct residual
// race), at a leaf the bonus from p_u.  Up to 64 nodes.
// The tree's streaming pass: the chain's, except that the draft row of a
// leaf (a node no other node hangs from) is neither loaded nor reduced.
template <int DT> struct TreeOp : ChainOp<DT> {
    static constexpr bool SKIPS = true;
    // bf16: items of 16 blocks (32 KB) on two CTAs per SM.  Measured against
    // 8-block items on four (same-box A/B, B = 64): k21 tree 183 -> 170 us,
    // w4 160 -> 148 us, 63-node tree 445 -> 396 us; the chain and greedy
    // streams keep 8-block items (both slower with 16).
    static constexpr int CTAS_PER_SM = 2;
    static constexpr int ITEM_BLOCKS = DT == 0 ? 8 : 16;
    // bf16: items numbered over the rows read and handed out by the call's
    // counter (table below); fp32 keeps the static stride over all rows with
    // the skip vote.  Measured (same-box A/B, B = 64, V = 151,936): bf16 k21
    // 167 -> 155 us, w4 146 -> 138, 63-node tree 393 -> 363; fp32 k21 229 ->
    // 243 (the balanced stream itself ended later than the static one's
    // slowest CTA).
    static constexpr bool TABLE = DT == 1;

    // Draft rows: lane v holds the parents of nodes v and v + 32 (16 bits
    // each, 0xffff for none or the root).  Target rows: no load.
    __device__ static __forceinline__ int skip_key(const ChainParams &P, long long row, int lane)
    {
        const long long b = div_row(row, P.R);
        const int rho = static_cast<int>(row - b * P.R);
        if (rho < P.nt) return -1;
        const int32_t *pp = P.tree_parent + b * P.nt;
        const int p0 = lane < P.nt ? __ldg(&pp[lane]) : -1;
        const int p1 = lane + 32 < P.nt ? __ldg(&pp[lane + 32]) : -1;
        return (p0 & 0xffff) | (p1 << 16);
    }

    __device__ static __forceinline__ bool skip(const ChainParams &P, long long row, int key, int)
    {
        const long long b = div_row(row, P.R);
        const int u = static_cast<int>(row - b * P.R) - P.nt;
        if (u < 0) return false;
        const bool hit = (key & 0xffff) == u || ((key >> 16) & 0xffff) == u;
        return __ballot_sync(0xffffffffu, hit) == 0u;
    }

    // The rows read, numbered (at most SKIP_TABLE_MAX sequences; built by the
    // whole CTA before the stream starts): bit u of mask[b] is set when node
    // u of sequence b is the parent of some node (then its draft row is read:
    // the same rows as the skip vote above), and first[b] counts the rows
    // that sequences 0 .. b-1 read (first[B]: all of them).  A sequence reads
    // its N target rows, then the draft rows of its set bits in node order.
    __device__ static void build_table(const ChainParams &P, unsigned long long *mask, int *first)
    {
        for (int b = threadIdx.x; b < P.B; b += blockDim.x) mask[b] = 0ull;
        __syncthreads();
        const int n = P.B * P.nt;
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            const int p = __ldg(&P.tree_parent[i]);
            if (p >= 0 && p < P.nt) atomicOr(&mask[i / P.nt], 1ull << p);
        }
        __syncthreads();
        if (threadIdx.x < 32) {  // exclusive prefix sum of the rows read, 32 sequences at a time
            const int lane = threadIdx.x;
            int run = 0;
            for (int base = 0; base < P.B; base += 32) {
                const int b = base + lane;
                const int cnt = b < P.B ? P.nt + __popcll(mask[b]) : 0;
                int incl = cnt;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int v = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += v;
                }
                if (b < P.B) first[b] = run + incl - cnt;
                run += __shfl_sync(0xffffffffu, incl, 31);
            }
            if (lane == 0) first[P.B] = run;
        }
        __syncthreads();
    }

    // Item `it` of the rows read: its row and chunk (binary search for the
    // sequence, then the k-th row read within it).
    __device__ static __forceinline__ void item_row(const ChainParams &P, const unsigned long long *mask,
                                                    const int *first, long long it, int nc, long long &row, int &c)
    {
        const int r = static_cast<int>(div_row(it, nc));
        c = static_cast<int>(it - static_cast<long long>(r) * nc);
        int lo = 0, hi = P.B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (first[mid] <= r) lo = mid;
            else hi = mid - 1;
        }
        const int k = r - first[lo];
        int rho = k;
        if (k >= P.nt) {
            unsigned long long m = mask[lo];
            for (int j = k - P.nt; j > 0; --j) m &= m - 1ull;
            rho = P.nt + __ffsll(static_cast<long long>(m)) - 1;
        }
        row = static_cast<long long>(lo) * P.R + rho;
    }

    // Before the finalize grid (which waits for this grid) meets in its
    // barriers: every sequence's barrier count and generation start at 0.
    __device__ static __forceinline__ void reset(const ChainParams &P)
    {
        if (blockIdx.x == 0 && P.tree_bar)
            for (int i = threadIdx.x; i < 2 * P.B; i += blockDim.x) P.tree_bar[i] = 0u;
    }
};

template <int DT, int FWV> struct TreeFin : ChainFin<DT, FWV> {
    using Fin = ChainFin<DT, FWV>;
    using Base = ChainOp<DT>;
    using Params = ChainParams;
    using Smem = ChainSmem;
    static constexpr int FIN_WARPS = FWV;
    static constexpr int FIN_BUF_FLOATS = 2 * FWV * G;

    __device__ static void write_bad_tree(const Params &P, int b, int rank, int lane)
    {
        const int N = P.nt;
        if (rank == 0 && threadIdx.x < 32) {
            for (int i = lane; i < N; i += 32) {
                P.out_tokens[static_cast<size_t>(b) * N + i] = -1;
                if (P.tree_nodes) P.tree_nodes[static_cast<size_t>(b) * N + i] = -1;
            }
            if (lane == 0) {
                P.accept_count[b] = -1;
                if (P.row_status) P.row_status[b] = STATUS_BAD_ROW;
            }
        }
    }

    // Coefficients of one residual pass: p(x) = ex2(z c2 - mt) ps and
    // q(x) = ex2(z' c2 - md) qs, with mt = Mt c2 rounded and its rounding
    // (delta = Mt c2 - mt, exact by FMA) folded into ps as 2^-delta, likewise
    // for the draft row, whose scale also carries the weight s.  One FFMA and
    // one ex2 per probability; identical target and draft rows still give
    // exactly p = q at s = 1.
    struct ResidCoef {
        float c2, mt, md, ps, qs;
    };

    __device__ static __forceinline__ ResidCoef resid_coef(const Params &P, float Mt, float St, float Md, float Sd,
                                                           float s)
    {
        constexpr float LN2 = 0.6931471805599453f;
        ResidCoef c;
        c.c2 = P.c2;
        c.mt = Mt * P.c2;
        c.md = Md * P.c2;
        const float dt = fmaf(Mt, P.c2, -c.mt), dd = fmaf(Md, P.c2, -c.md);
        c.ps = __fmul_rn(1.f / St, fmaf(-dt, LN2, 1.f));
        c.qs = __fmul_rn(__fmul_rn(1.f / Sd, fmaf(-dd, LN2, 1.f)), s);
        return c;
    }

    __device__ static __forceinline__ float rterm(float zt, float zd, const ResidCoef &c)
    {
        // (zt, zd) as a packed pair: one FMA for both exponent arguments and
        // one multiply for both scales, each element rounded as alone
        float at, ad, p, q;
        unpack2(ffma2(pack2(zt, zd), pack2(c.c2, c.c2), pack2(-c.mt, -c.md)), at, ad);
        unpack2(mul2(pack2(fast_exp2(at), fast_exp2(ad)), pack2(c.ps, c.qs)), p, q);
        return fmaxf(__fsub_rn(p, q), 0.f);
    }

    // Residual mass of block beta, sum over x of max(0, p(x) - s q(x)) (this
    // lane's share); 16-byte loads when the rows are 16-byte aligned, the
    // ragged tail padded with -inf logits (mass 0).
    __device__ static __forceinline__ float block_resid(const Params &P, const unsigned char *tp,
                                                        const unsigned char *dp, int beta, const ResidCoef &rc,
                                                        int lane)
    {
        const int lo = beta * G, hi = min(P.V, lo + G);
        float pa[4] = {0.f, 0.f, 0.f, 0.f};
        if (P.vec) {
            if constexpr (DT == 0) {
                const float4 *t4 = reinterpret_cast<const float4 *>(tp) + lo / 4;
                const float4 *d4 = reinterpret_cast<const float4 *>(dp) + lo / 4;
                const int n4 = (hi - lo) >> 2;
#pragma unroll
                for (int h = 0; h < G / 512; ++h) {
                    float4 a[4], c[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int i = lane + 32 * (4 * h + j);
                        if (i < n4) {
                            a[j] = __ldcg(t4 + i);
                            c[j] = __ldcg(d4 + i);
                        } else {
                            a[j] = c[j] = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        pa[0] += rterm(a[j].x, c[j].x, rc);
                        pa[1] += rterm(a[j].y, c[j].y, rc);
                        pa[2] += rterm(a[j].z, c[j].z, rc);
                        pa[3] += rterm(a[j].w, c[j].w, rc);
                    }
                }
            } else {
                const uint4 *t8 = reinterpret_cast<const uint4 *>(tp) + lo / 8;
                const uint4 *d8 = reinterpret_cast<const uint4 *>(dp) + lo / 8;
                const int n8 = (hi - lo) >> 3;
                constexpr unsigned NEG = 0xff80ff80u;  // two bf16 -inf
                uint4 a[G / 256], c[G / 256];
#pragma unroll
                for (int j = 0; j < G / 256; ++j) {
                    const int i = lane + 32 * j;
                    if (i < n8) {
                        a[j] = __ldcg(t8 + i);
                        c[j] = __ldcg(d8 + i);
                    } else {
                        a[j] = c[j] = make_uint4(NEG, NEG, NEG, NEG);
                    }
                }
#pragma unroll
                for (int j = 0; j < G / 256; ++j) {
                    const unsigned wa[4] = {a[j].x, a[j].y, a[j].z, a[j].w}, wc[4] = {c[j].x, c[j].y, c[j].z, c[j].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        pa[e] += rterm(__uint_as_float(wa[e] << 16), __uint_as_float(wc[e] << 16), rc);
                        pa[e] += rterm(__uint_as_float(wa[e] & 0xffff0000u), __uint_as_float(wc[e] & 0xffff0000u), rc);
                    }
                }
            }
        } else {
            for (int x = lo + lane; x < hi; x += 32)
                pa[0] += rterm(DType<DT>::load(tp, x), DType<DT>::load(dp, x), rc);
        }
        return (pa[0] + pa[1]) + (pa[2] + pa[3]);
    }

    // One warp's blocks of a residual pass over 16-byte aligned rows, in
    // units of 2 KB of each row (a bf16 block, half an fp32 block): each lane
    // copies its own four 16-byte pieces of both rows into one of two 4 KB
    // stages of the warp's buffer (cp.async), the next unit's while it sums
    // this one, and reads back only what it copied itself (no warp barrier).
    __device__ static void pass_async(const Params &P, float *rb, int first, int stride, const unsigned char *tp,
                                      const unsigned char *dp, const ResidCoef &rc, unsigned char *buf, int lane)
    {
        constexpr int EB = DType<DT>::BYTES, UE = 2048 / EB, UPB = G / UE, PER = 16 / EB;
        const int nblk = first < P.nb ? (P.nb - 1 - first) / stride + 1 : 0;
        const int U = nblk * UPB;
        auto unit_e0 = [&](int u, int &beta) {
            const int i = u / UPB;
            beta = first + i * stride;
            return beta * G + (u - i * UPB) * UE;
        };
        auto issue = [&](int u) {
            int beta;
            const int e0 = unit_e0(u, beta);
            const int n = min(UE, P.V - e0);
            unsigned char *st = buf + (u & 1) * 4096;
            const unsigned char *ts = tp + static_cast<size_t>(e0) * EB, *ds = dp + static_cast<size_t>(e0) * EB;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int i = lane + 32 * j;
                if (i * PER < n) {
                    cp_async16(st + 16 * i, ts + 16 * i);
                    cp_async16(st + 2048 + 16 * i, ds + 16 * i);
                }
            }
            cp_async_commit();
        };
        float pa[4] = {0.f, 0.f, 0.f, 0.f};
        if (U > 0) issue(0);
        for (int u = 0; u < U; ++u) {
            if (u + 1 < U) {
                issue(u + 1);
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
            int beta;
            const int e0 = unit_e0(u, beta);
            const int n = min(UE, P.V - e0);
            const unsigned char *st = buf + (u & 1) * 4096;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int i = lane + 32 * j;
                if (i * PER < n) {
                    if constexpr (DT == 0) {
                        const float4 a = reinterpret_cast<const float4 *>(st)[i];
                        const float4 c = reinterpret_cast<const float4 *>(st + 2048)[i];
                        pa[0] += rterm(a.x, c.x, rc);
                        pa[1] += rterm(a.y, c.y, rc);
                        pa[2] += rterm(a.z, c.z, rc);
                        pa[3] += rterm(a.w, c.w, rc);
                    } else {
                        const uint4 a = reinterpret_cast<const uint4 *>(st)[i];
                        const uint4 c = reinterpret_cast<const uint4 *>(st + 2048)[i];
                        const unsigned wa[4] = {a.x, a.y, a.z, a.w}, wc[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            pa[e] += rterm(__uint_as_float(wa[e] << 16), __uint_as_float(wc[e] << 16), rc);
                            pa[e] += rterm(__uint_as_float(wa[e] & 0xffff0000u), __uint_as_float(wc[e] & 0xffff0000u), rc);
                        }
                    }
                }
            }
            if ((u + 1) % UPB == 0) {
                const float part = warp_sum((pa[0] + pa[1]) + (pa[2] + pa[3]));
                if (lane == 0) rb[beta] = part;
                pa[0] = pa[1] = pa[2] = pa[3] = 0.f;
            }
        }
    }

    // Residual pass j of sequence b: the block masses of max(0, p_u - s q_u),
    // the blocks split over the sequence's cs CTAs (buffer j % 2, so a pass
    // never overwrites masses another CTA may still be summing), then in
    // every CTA N = their sum in one fixed order (identical in all of them).
    __device__ static bool tree_pass(const Params &P, int b, int rank, int j, const unsigned char *tp,
                                     const unsigned char *dp, float Mt, float St, float Md, float Sd, float s, Smem &sm,
                                     unsigned char *buf, int warp, int lane)
    {
        float *rb = P.resid + (static_cast<size_t>(b) * 2 + (j & 1)) * P.nb;
        const ResidCoef rc = resid_coef(P, Mt, St, Md, Sd, s);
        // bf16 rows through the copy pipeline below; fp32 rows with plain
        // loads, a block at a time (measured: the pipeline takes the k21 bf16
        // call from 155.7 to 154.1 us and the fp32 one from 228 to 230 us)
        if (DT == 1 && P.vec) {
            pass_async(P, rb, rank * FWV + warp, P.cs * FWV, tp, dp, rc, buf, lane);
        } else {
            for (int beta = rank * FWV + warp; beta < P.nb; beta += P.cs * FWV) {
                const float part = warp_sum(block_resid(P, tp, dp, beta, rc, lane));
                if (lane == 0) rb[beta] = part;
            }
        }
        if (lane == 0) __threadfence();  // this warp's masses, before the barrier's arrival
        bool ok = true;
        if (P.cs > 1)
            ok = group_barrier<FWV * 32>(P.tree_bar + 2 * b, static_cast<unsigned>(P.cs), static_cast<unsigned>(j),
                                         P.err, &sm.gflag);
        else
            fin_sync<FWV>();
        if (!ok) return false;
        if (warp == 0) {
            float z = 0.f;
            for (int beta = lane; beta < P.nb; beta += 32) z += __ldcg(&rb[beta]);
            z = warp_sum(z);
            if (lane == 0) sm.Z = z;
        }
        fin_sync<FWV>();
        return true;
    }

    // Group g = b * cs + rank: CTA `rank` of sequence b.  Every CTA of the
    // sequence walks the tree and takes the same decisions from the same
    // values; rank 0 writes the outputs.
    __device__ static void finalize(const Params &P, int g, Smem &sm, float *buf, int warp, int lane)
    {
        const int b = g / P.cs, rank = g - b * P.cs;
        const int N = P.nt, nb = P.nb;
        float *tb = buf + warp * 2 * G, *db = tb + G;
        // A. Inputs: parents, tokens, uniforms, and each node's token logit
        //    in its parent's target and draft rows (before the dependent wait).
        if (threadIdx.x == 0) {
            sm.bad = 0;
            sm.key = P.keys[b];
            sm.cached = (N * nb <= STAT_CACHE) ? 1 : 0;
        }
        if (warp == 0) {
            for (int v = lane; v < N; v += 32) {
                const int pv = P.tree_parent[static_cast<size_t>(b) * N + v];
                const int x = P.tokens[static_cast<size_t>(b) * N + v];
                sm.par[v] = pv;
                sm.x[v] = x;
                sm.rr[v] = P.r[static_cast<size_t>(b) * N + v];
                const bool ok = (v == 0) ? (pv == -1) : (pv >= 0 && pv < v && x >= 0 && x < P.V);
                sm.zt[v] = sm.zd[v] = 0.f;
                if (v > 0 && ok) {
                    sm.zt[v] = DType<DT>::load(Base::row_of(P, b, pv), x);
                    sm.zd[v] = DType<DT>::load(Base::row_of(P, b, N + pv), x);
                }
                if (!ok) atomicOr(&sm.bad, 1);
            }
        }
        asm volatile("griddepcontrol.wait;" ::: "memory");
        fin_sync<FWV>();
        // B. Row statistics; a bad target row, or a bad draft row of a node
        //    with children, makes the sequence bad (a leaf's draft row was
        //    not streamed and is not looked at).
        Base::template merge_stats<FWV, true>(P, b, sm, N, false, warp, lane);
        fin_sync<FWV>();
        if (warp == 0 && !sm.bad) {
            bool bad = false;
            for (int v = lane; v < N; v += 32) {
                if (!(sm.S[v] > 0.f)) bad = true;                           // target row of v
                if (v > 0 && !(sm.S[N + sm.par[v]] > 0.f)) bad = true;      // draft row of v's parent
            }
            if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(&sm.bad, 1);
        }
        fin_sync<FWV>();
        if (sm.bad) {
            write_bad_tree(P, b, rank, lane);
            return;
        }
        // C. The walk.
        const uint64_t key = sm.key;
        int u = 0, k = 0, res = -1, pass = 0;
        for (;;) {
            const unsigned long long kids =
                static_cast<unsigned long long>(__ballot_sync(0xffffffffu, lane < N && lane > u && sm.par[lane] == u)) |
                (static_cast<unsigned long long>(
                     __ballot_sync(0xffffffffu, lane + 32 < N && lane + 32 > u && sm.par[lane + 32] == u))
                 << 32);
            const float Mt = sm.M[u], St = sm.S[u];
            const unsigned char *tp = Base::row_of(P, b, u);
            if (kids == 0ull) {
                // leaf: the bonus token from p_u (warp 0)
                if (warp == 0) {
                    DrawVariates dv;
                    draw_variates(dv, key, 0u, nb, lane);
                    const int beta = Base::race_blocks_p(P, sm, b, u, Mt, key, 0u, lane, dv, true);
                    Base::load_block(P, tp, beta, tb, lane);
                    const int x = Base::race_in_block_p(P, tb, beta, Base::block_max(P, sm, b, u, beta), dv, lane);
                    if (lane == 0) sm.result = x;
                }
                fin_sync<FWV>();
                res = sm.result;
                break;
            }
            const float Md = sm.M[N + u], Sd = sm.S[N + u];
            const unsigned char *dp = Base::row_of(P, b, N + u);
            float sres = 0.f, Nm = 1.f;
            int next = -1;
            for (unsigned long long m = kids; m; m &= m - 1ull) {
                const int c = __ffsll(static_cast<long long>(m)) - 1;
                const float px = expf((sm.zt[c] - Mt) * P.invT) / St;
                const float qx = expf((sm.zd[c] - Md) * P.invT) / Sd;
                float Pm = px;
                if (sres > 0.f) {
                    const float d = __fsub_rn(px, __fmul_rn(sres, qx));
                    Pm = d > 0.f ? d / Nm : 0.f;
                }
                if (Pm > 0.f && sm.rr[c] * qx <= Pm) {
                    next = c;
                    break;
                }
                // rejected: the next residual.  Its mass N_m is needed for the
                // next child's test; after the last child the draw below
                // needs only s (the pass runs there if the trials all fail).
                sres += Nm;
                if ((m & (m - 1ull)) == 0ull) break;
                if (!tree_pass(P, b, rank, pass++, tp, dp, Mt, St, Md, Sd, sres, sm, reinterpret_cast<unsigned char *>(tb), warp, lane)) {
                    write_bad_tree(P, b, rank, lane);  // a CTA of the sequence did not arrive (error flag set)
                    return;
                }
                Nm = sm.Z;
                if (!(Nm > 0.f)) {  // no residual mass (a token outside q's support)
                    write_bad_tree(P, b, rank, lane);
                    return;
                }
            }
            if (next >= 0) {
                if (rank == 0 && threadIdx.x == 0) {
                    P.out_tokens[static_cast<size_t>(b) * N + k] = sm.x[next];
                    if (P.tree_nodes) P.tree_nodes[static_cast<size_t>(b) * N + k] = next;
                }
                ++k;
                u = next;
                continue;
            }
            // every child rejected: one draw from max(0, p_u - s q_u), FWV trials per round
            if (threadIdx.x == 0) sm.result = -1;
            fin_sync<FWV>();
            for (int round = 0; round < MAX_TRIALS / FWV; ++round) {
                const uint32_t t = static_cast<uint32_t>(round * FWV + warp);
                DrawVariates dv;
                draw_variates(dv, key, t, nb, lane);
                const int beta = Base::race_blocks_p(P, sm, b, u, Mt, key, t, lane, dv, true);
                Base::load_block(P, tp, beta, tb, lane);
                Base::load_block(P, dp, beta, db, lane);
                const int x = Base::race_in_block_p(P, tb, beta, Base::block_max(P, sm, b, u, beta), dv, lane);
                if (lane == 0) {
                    const float v = uniform24(dv.aw);
                    const float p = expf((tb[x - beta * G] - Mt) * P.invT) / St;
                    const float q = __fmul_rn(expf((db[x - beta * G] - Md) * P.invT) / Sd, sres);
                    sm.trial_x[0][warp] = x;
                    sm.trial_acc[0][warp] = (q <= (1.0f - v) * p) ? 1 : 0;
                }
                fin_sync<FWV>();
                if (threadIdx.x == 0) {
                    for (int w = 0; w < FWV; ++w)
                        if (sm.trial_acc[0][w]) {
                            sm.result = sm.trial_x[0][w];
                            break;
                        }
                }
                fin_sync<FWV>();
                if (sm.result >= 0) break;
            }
            if (sm.result < 0) {
                // the direct draw: block masses of max(0, p_u - s q_u) (no
                // mass at all leaves nothing to draw: bad row, below)
                if (!tree_pass(P, b, rank, pass++, tp, dp, Mt, St, Md, Sd, sres, sm, reinterpret_cast<unsigned char *>(tb), warp, lane)) {
                    write_bad_tree(P, b, rank, lane);
                    return;
                }
                if (warp == 0) {
                    const float *rb = P.resid + (static_cast<size_t>(b) * 2 + ((pass - 1) & 1)) * nb;
                    const int x = Base::race_resid(P, b, tp, dp, Mt, St, Md, Sd, key, tb, db, nullptr, sres, lane, rb);
                    if (lane == 0) sm.result = x;
                }
                fin_sync<FWV>();
            }
            res = sm.result;
            break;
        }
        if (res < 0) {
            write_bad_tree(P, b, rank, lane);
            return;
        }
        if (rank == 0 && threadIdx.x < 32) {
            for (int i = k + lane; i < N; i += 32) {
                P.out_tokens[static_cast<size_t>(b) * N + i] = (i == k) ? res : -1;
                if (P.tree_nodes) P.tree_nodes[static_cast<size_t>(b) * N + i] = -1;
            }
            if (lane == 0) {
                P.accept_count[b] = k;
                if (P.row_status) P.row_status[b] = 0;
            }
        }
    }
};

// =====================================================================================
// Greedy verify, T = 0
// =====================================================================================
struct GreedyParams {
    long long total_items;
    int nc, nb, V;
    unsigned *err;
    const unsigned char *target;
    const int32_t *tokens;
    int B, gamma, R;  // R = gamma + 1
    int32_t *accept_count, *out_tokens, *row_status;
    int2 *best;  // [B*R*nb] (max value bits, argmax id); id -2 marks a bad block
    CacheLookup cache;
    const int32_t *tree_parent;  // greedy tree verify: [B, N] parents (R = N)
    int32_t *tree_nodes;
};

struct GreedySmem {
    int a[65];
    int x[64];
    int par[64];
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

    static constexpr int CTAS_PER_SM = DT == 0 ? 2 : 4;

    __device__ static __forceinline__ void block_smem(const Params &P, long long row, int beta,
                                                      const unsigned char *blk, int valid, int lane)
    {
        if constexpr (DT == 0) {
            float v[32];
            load_block_smem<DT>(v, blk, lane);
            mask_tail<DT>(v, valid, lane);
            block(P, row, beta, v, valid, lane);
        } else {
            block_bf16(P, row, beta, blk, valid, lane);
        }
    }

    // bf16 from the staged block, packed: the block max by bf16x2 max with
    // NaN propagation, then the first id holding it (ids rise with the word
    // index within a lane, so the first match is the smallest; -0.0 == +0.0).
    __device__ static __forceinline__ void block_bf16(const Params &P, long long row, int beta,
                                                      const unsigned char *blk, int valid, int lane)
    {
        uint32_t w[16];
        const uint4 *p = reinterpret_cast<const uint4 *>(blk);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 t = p[j * 32 + lane];
            w[4 * j] = t.x;
            w[4 * j + 1] = t.y;
            w[4 * j + 2] = t.z;
            w[4 * j + 3] = t.w;
        }
        if (valid < G) {  // element 2h / 2h+1 of word h of vector j: j*256 + lane*8 + 2h (+1)
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const int e0 = (q >> 2) * 256 + lane * 8 + 2 * (q & 3);
                if (e0 >= valid) w[q] = (w[q] & 0xffff0000u) | 0xff80u;
                if (e0 + 1 >= valid) w[q] = (w[q] & 0x0000ffffu) | 0xff800000u;
            }
        }
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(w);
        __nv_bfloat162 mx[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) mx[a] = __hmax2_nan(h[a], h[a + 8]);
#pragma unroll
        for (int a = 0; a < 4; ++a) mx[a] = __hmax2_nan(mx[a], mx[a + 4]);
        mx[0] = __hmax2_nan(__hmax2_nan(mx[0], mx[1]), __hmax2_nan(mx[2], mx[3]));
        const float lo = __low2float(mx[0]), hi = __high2float(mx[0]);
        const bool nan = __any_sync(0xffffffffu, isnan(lo) || isnan(hi));
        const float m = warp_max_redux(fmaxf(lo, hi));
        int i = INT_MAX;
        if (!nan && m != -INFINITY && m != INFINITY) {
            const __nv_bfloat162 mm = __float2bfloat162_rn(m);  // exact: m is one of the bf16 values
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const unsigned e = __heq2_mask(h[q], mm);
                const int id0 = (q >> 2) * 256 + lane * 8 + 2 * (q & 3);
                const int c = (e & 0xffffu) ? id0 : ((e >> 16) ? id0 + 1 : INT_MAX);
                i = min(i, c);
            }
            i = static_cast<int>(__reduce_min_sync(0xffffffffu, static_cast<unsigned>(i)));
        }
        if (lane == 0) {
            int2 o;
            if (nan || m == INFINITY) o = make_int2(0x7fc00000, -2);
            else o = make_int2(__float_as_int(m), i == INT_MAX ? INT_MAX : beta * G + i);
            P.best[row * P.nb + beta] = o;
        }
    }

    // Per-block (max, first argmax): four independent accumulators over the
    // lane's elements e = a (mod 4), each in rising id order, then combined
    // with ties to the lower id.
    __device__ static __forceinline__ void block(const Params &P, long long row, int beta, float v[32], int, int lane)
    {
        float bv[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        int bi[4] = {INT_MAX, INT_MAX, INT_MAX, INT_MAX};
        bool nan = false;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            const float x = v[e];
            nan |= (x != x);
            if (x > bv[e & 3]) {  // strict: the first (lowest) id keeps a tie; -0.0 == +0.0
                bv[e & 3] = x;
                bi[e & 3] = lane_index<DT>(lane, e);
            }
        }
        float b = bv[0];
        int i = bi[0];
#pragma unroll
        for (int a = 1; a < 4; ++a)
            if (bv[a] > b || (bv[a] == b && bi[a] < i)) {
                b = bv[a];
                i = bi[a];
            }
        warp_argmax(b, i);
        nan = __any_sync(0xffffffffu, nan);
        if (lane == 0) {
            int2 o;
            if (nan || b == INFINITY) o = make_int2(0x7fc00000, -2);
            else o = make_int2(__float_as_int(b), i == INT_MAX ? INT_MAX : beta * G + i);
            P.best[row * P.nb + beta] = o;
        }
    }

    static constexpr int FIN_WARPS = NCW;
    static constexpr int FIN_BUF_FLOATS = 0;

    __device__ static void finalize(const Params &P, int b, Smem &sm, float *, int warp, int lane)
    {
        const int g = P.gamma, R = P.R, nb = P.nb;
        if (threadIdx.x == 0) sm.bad = 0;
        if (warp == 0 && lane < g) sm.x[lane] = P.tokens[static_cast<size_t>(b) * g + lane];
        if (warp == 1) cache_prefetch(P.cache, b, lane);
        asm volatile("griddepcontrol.wait;" ::: "memory");
        consumer_sync();
        if (warp == 0 && lane < g && (sm.x[lane] < 0 || sm.x[lane] >= P.V)) atomicOr(&sm.bad, 1);
        if (threadIdx.x == 32 && workspace_timed_out(P.err)) atomicOr(&sm.bad, 2);  // block results incomplete
        for (int rho = warp; rho < R; rho += NCW) {
            const int2 *bb = P.best + (static_cast<long long>(b) * R + rho) * nb;
            float bv = -INFINITY;
            int bi = INT_MAX;
            bool bad = false;
            for (int base = 0; base < nb; base += 32 * 8) {
                int2 o[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int beta = base + 32 * u + lane;
                    o[u] = beta < nb ? __ldcg(&bb[beta]) : make_int2(__float_as_int(-INFINITY), INT_MAX);
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    if (o[u].y == -2) {
                        bad = true;
                    } else {
                        const float v = __int_as_float(o[u].x);
                        if (v > bv || (v == bv && o[u].y < bi)) {
                            bv = v;
                            bi = o[u].y;
                        }
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
        consumer_sync();
        if (warp == 0) {
            if (sm.bad) {
                for (int i = lane; i <= g; i += 32) P.out_tokens[static_cast<size_t>(b) * (g + 1) + i] = -1;
                if (lane == 0) {
                    P.accept_count[b] = -1;
                    if (P.row_status) P.row_status[b] = (sm.bad & 2) ? STATUS_TIMEOUT : STATUS_BAD_ROW;
                }
                cache_lookup(P.cache, b, -1, -1, lane);
            } else {
                const bool acc = lane < g && sm.x[lane] == sm.a[lane];
                const unsigned mask = __ballot_sync(0xffffffffu, acc);
                const unsigned all = (g == 32) ? 0xffffffffu : ((1u << g) - 1u);
                const int k = ((mask & all) == all) ? g : (__ffs(~mask) - 1);
                for (int i = lane; i <= g; i += 32) {
                    int v = -1;
                    if (i < k) v = sm.x[i];
                    else if (i == k) v = sm.a[k];
                    P.out_tokens[static_cast<size_t>(b) * (g + 1) + i] = v;
                }
                if (lane == 0) {
                    P.accept_count[b] = k;
                    if (P.row_status) P.row_status[b] = 0;
                }
                cache_lookup(P.cache, b, k, sm.a[k], lane);
            }
        }
    }
};

// Greedy tree verify (T = 0): descend into the first child whose token is
// the argmax of p_u (lowest id on ties); emit the argmax of the last node.
template <int DT> struct GreedyTreeFin : GreedyOp<DT> {
    using Params = GreedyParams;
    using Smem = GreedySmem;
    static constexpr int FIN_WARPS = NCW;
    static constexpr int FIN_BUF_FLOATS = 0;

    __device__ static void finalize(const Params &P, int b, Smem &sm, float *, int warp, int lane)
    {
        const int N = P.R, nb = P.nb;
        if (threadIdx.x == 0) sm.bad = 0;
        if (warp == 0) {
            for (int v = lane; v < N; v += 32) {
                const int pv = P.tree_parent[static_cast<size_t>(b) * N + v];
                const int x = P.tokens[static_cast<size_t>(b) * N + v];
                sm.par[v] = pv;
                sm.x[v] = x;
                const bool ok = (v == 0) ? (pv == -1) : (pv >= 0 && pv < v && x >= 0 && x < P.V);
                if (!ok) atomicOr(&sm.bad, 1);
            }
        }
        asm volatile("griddepcontrol.wait;" ::: "memory");
        consumer_sync();
        for (int rho = warp; rho < N; rho += NCW) {
            const int2 *bb = P.best + (static_cast<long long>(b) * N + rho) * nb;
            float bv = -INFINITY;
            int bi = INT_MAX;
            bool bad = false;
            for (int beta = lane; beta < nb; beta += 32) {
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
        consumer_sync();
        if (warp != 0) return;
        if (sm.bad) {
            for (int i = lane; i < N; i += 32) {
                P.out_tokens[static_cast<size_t>(b) * N + i] = -1;
                if (P.tree_nodes) P.tree_nodes[static_cast<size_t>(b) * N + i] = -1;
            }
            if (lane == 0) {
                P.accept_count[b] = -1;
                if (P.row_status) P.row_status[b] = STATUS_BAD_ROW;
            }
            return;
        }
        int u = 0, k = 0;
        for (;;) {
            const int au = sm.a[u];
            const unsigned m0 = __ballot_sync(0xffffffffu, lane < N && lane > u && sm.par[lane] == u && sm.x[lane] == au);
            const int w = lane + 32;
            const unsigned m1 = __ballot_sync(0xffffffffu, w < N && w > u && sm.par[w] == u && sm.x[w] == au);
            if (!m0 && !m1) break;
            const int c = m0 ? __ffs(m0) - 1 : 32 + __ffs(m1) - 1;
            if (lane == 0) {
                P.out_tokens[static_cast<size_t>(b) * N + k] = sm.x[c];
                if (P.tree_nodes) P.tree_nodes[static_cast<size_t>(b) * N + k] = c;
            }
            ++k;
            u = c;
        }
        for (int i = k + lane; i < N; i += 32) {
            P.out_tokens[static_cast<size_t>(b) * N + i] = (i == k) ? sm.a[u] : -1;
            if (P.tree_nodes) P.tree_nodes[static_cast<size_t>(b) * N + i] = -1;
        }
        if (lane == 0) {
            P.accept_count[b] = k;
            if (P.row_status) P.row_status[b] = 0;
        }
    }
};

// =====================================================================================
// Host launch
// =====================================================================================
size_t chain_ws_bytes(int B, int gamma, int V)
{
    const size_t nb = blocks_per_row(V), R = 2 * static_cast<size_t>(gamma) + 1;
    size_t n = WS_HEADER;
    n += align256(static_cast<size_t>(B) * R * nb * 8); // block statistics
    n += align256(static_cast<size_t>(B) * nb * 4);  // residual block masses
    const size_t gr = greedy_ws_bytes(B, gamma, V);
    return n > gr ? n : gr;
}

size_t greedy_ws_bytes(int B, int gamma, int V)
{
    const size_t nb = blocks_per_row(V), R = static_cast<size_t>(gamma) + 1;
    return WS_HEADER + align256(static_cast<size_t>(B) * R * nb * 8);
}

// Offsets of the fan-out positions in a sequence's candidate row.
static void fill_cache(CacheLookup &C, const ChainLaunch &L)
{
    C.ids = L.cache_ids;
    C.slot = L.cache_slot;
    C.n = 0;
    if (!L.cache_ids) return;
    for (int k = 0; k <= L.gamma; ++k) {
        C.off[k] = C.n;
        C.n += L.cache_fanout[k];
    }
    C.off[L.gamma + 1] = C.n;
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
    P.nt = L.gamma + 1;
    P.nd = L.gamma;
    P.total_items = static_cast<long long>(L.B) * P.R * P.nc;
    unsigned char *ws = static_cast<unsigned char *>(L.ws);
    P.err = reinterpret_cast<unsigned *>(ws);
    size_t off = WS_HEADER;
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
    P.vec = L.tma ? 1 : 0;
    P.accept_count = L.accept_count;
    P.out_tokens = L.out_tokens;
    P.out_pq = L.out_pq;
    P.out_Z = L.out_Z;
    P.row_status = L.row_status;
    fill_cache(P.cache, L);
    P.sag = L.sag;
    P.invC = L.sag ? 1.0f / L.sag_C : 1.0f;
    // One finalize CTA per sequence.  While the sequences fit on the SMs at
    // once: the 16-warp CTA (16 residual trials per round) for fp32 batches
    // above 32, else the 8-warp CTA; both draw the first round's variates
    // before the dependent-grid wait.  Measured (same-box A/B against the
    // 16-warp CTA everywhere): 8 warps for bf16 B = 64 -2.7 %, spd gamma = 1
    // -5.6 %, fp32 B = 8 -8 %, B = 1 -15 %, but fp32 B = 64 +0.1 to +1.2 %
    // (a smaller CTA starts sooner after the stream; fewer trials per round
    // more often need a second round).  Beyond the SM count: the 8-warp CTA
    // without the parked variates, two per SM.
    int sms = 0;
    cudaError_t e = device_sm_count(&sms);
    if (e != cudaSuccess) return e;
    const bool fits = L.B <= sms;
    if (L.dtype == 0) {
        if (fits && L.B > 32) return launch_stream_finalize<ChainOp<0>, ChainFin<0, FW>, 0>(P, L.tma, L.B, st);
        return fits ? launch_stream_finalize<ChainOp<0>, ChainFin<0, NCW, true>, 0>(P, L.tma, L.B, st)
                    : launch_stream_finalize<ChainOp<0>, ChainFin<0, NCW>, 0>(P, L.tma, L.B, st);
    }
    return fits ? launch_stream_finalize<ChainOp<1>, ChainFin<1, NCW, true>, 1>(P, L.tma, L.B, st)
                : launch_stream_finalize<ChainOp<1>, ChainFin<1, NCW>, 1>(P, L.tma, L.B, st);
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
    P.best = reinterpret_cast<int2 *>(ws + WS_HEADER);
    P.target = static_cast<const unsigned char *>(L.target);
    P.tokens = L.tokens;
    P.accept_count = L.accept_count;
    P.out_tokens = L.out_tokens;
    P.row_status = L.row_status;
    fill_cache(P.cache, L);
    return L.dtype == 0 ? launch_stream_finalize<GreedyOp<0>, GreedyOp<0>, 0>(P, L.tma, L.B, st)
                        : launch_stream_finalize<GreedyOp<1>, GreedyOp<1>, 1>(P, L.tma, L.B, st);
}

size_t tree_ws_bytes(int B, int N, int V)
{
    const size_t nb = blocks_per_row(V), R = 2 * static_cast<size_t>(N);
    size_t n = WS_HEADER;
    n += align256(static_cast<size_t>(B) * R * nb * 8);  // block statistics
    n += align256(static_cast<size_t>(B) * 2 * nb * 4);  // residual block masses, two buffers
    n += align256(static_cast<size_t>(B) * 2 * 4);       // barrier of each sequence's finalize CTAs
    const size_t gr = WS_HEADER + align256(static_cast<size_t>(B) * N * nb * 8);
    return n > gr ? n : gr;
}

cudaError_t launch_tree(const TreeLaunch &L, cudaStream_t st)
{
    unsigned char *ws = static_cast<unsigned char *>(L.ws);
    if (L.T == 0.0f) {
        GreedyParams P{};
        P.V = L.V;
        P.nb = blocks_per_row(L.V);
        P.nc = chunks_per_row(L.V);
        P.B = L.B;
        P.gamma = L.N - 1;
        P.R = L.N;
        P.total_items = static_cast<long long>(L.B) * P.R * P.nc;
        P.err = reinterpret_cast<unsigned *>(ws);
        P.best = reinterpret_cast<int2 *>(ws + WS_HEADER);
        P.target = static_cast<const unsigned char *>(L.target);
        P.tokens = L.tokens;
        P.accept_count = L.accept_count;
        P.out_tokens = L.out_tokens;
        P.row_status = L.row_status;
        P.tree_parent = L.parent;
        P.tree_nodes = L.out_nodes;
        return L.dtype == 0 ? launch_stream_finalize<GreedyOp<0>, GreedyTreeFin<0>, 0>(P, L.tma, L.B, st)
                            : launch_stream_finalize<GreedyOp<1>, GreedyTreeFin<1>, 1>(P, L.tma, L.B, st);
    }
    ChainParams P{};
    P.V = L.V;
    P.nb = blocks_per_row(L.V);
    P.nc = chunks_per_row(L.V);
    P.B = L.B;
    P.gamma = L.N - 1;
    P.nt = L.N;
    P.nd = L.N;
    P.R = 2 * L.N;
    P.total_items = static_cast<long long>(L.B) * P.R * P.nc;
    P.err = reinterpret_cast<unsigned *>(ws);
    size_t off = WS_HEADER;
    P.stats = reinterpret_cast<float2 *>(ws + off);
    off += align256(static_cast<size_t>(L.B) * P.R * P.nb * 8);
    P.resid = reinterpret_cast<float *>(ws + off);
    off += align256(static_cast<size_t>(L.B) * 2 * P.nb * 4);
    P.tree_bar = reinterpret_cast<unsigned *>(ws + off);
    P.target = static_cast<const unsigned char *>(L.target);
    P.draft = static_cast<const unsigned char *>(L.draft);
    P.tokens = L.tokens;
    P.r = L.r;
    P.keys = L.keys;
    P.invT = 1.0f / L.T;
    P.c2 = 1.4426950408889634f / L.T;
    P.vec = L.tma ? 1 : 0;
    P.accept_count = L.accept_count;
    P.out_tokens = L.out_tokens;
    P.row_status = L.row_status;
    P.invC = 1.0f;
    P.tree_parent = L.parent;
    P.tree_nodes = L.out_nodes;
    int sms = 0;
    cudaError_t e = device_sm_count(&sms);
    if (e != cudaSuccess) return e;
    // The walk's residual passes (one per rejected child) are split over a
    // cluster of cs CTAs per sequence, as many as the idle SMs allow (<= 8).
    int cs = 1;
    while (cs < 8 && L.B * cs * 2 <= sms) cs *= 2;
    P.cs = cs;
    const bool wide = L.B <= sms;
    if (L.dtype == 0)
        return wide ? launch_stream_finalize<TreeOp<0>, TreeFin<0, FW>, 0>(P, L.tma, L.B * cs, st, cs)
                    : launch_stream_finalize<TreeOp<0>, TreeFin<0, NCW>, 0>(P, L.tma, L.B, st);
    return wide ? launch_stream_finalize<TreeOp<1>, TreeFin<1, FW>, 1>(P, L.tma, L.B * cs, st, cs)
                : launch_stream_finalize<TreeOp<1>, TreeFin<1, NCW>, 1>(P, L.tma, L.B, st);
}

}  // namespace spv
