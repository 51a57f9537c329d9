// spv_filtered.cu -- chain verify on top-k / top-p filtered distributions.
//
// "Speculative Pipeline Decoding", section "Evaluation": the sampled runs
// (T = 1) draw from target and draft distributions restricted to the top-k
// = 50 logits with top-p = 1.0.  The verify step of "Speculative Decoding:
// How Draft-Model Parallelism Cuts LLM Inference Latency" ("The four-phase
// loop", steps 3 and 4) then runs on those filtered distributions p', q':
// only the top_k logits of each of the 2 gamma + 1 rows matter.
//
// Three kernels per call, each row still read once in full:
//   1. sample (one warp per row): from eight evenly spaced 1024-logit blocks
//      of the row, the m-th largest of their 32-logit group maxima is a
//      threshold tau0 that m distinct logits reach; m is chosen so that about
//      3.5 k logits of the whole row are expected at or above it.
//   2. stream (the persistent streaming kernel): every logit is compared
//      with its row's tau0 (two instructions per logit: a max and a NaN/+inf
//      check); the few at or above it are appended to the row's candidate
//      buffer.
//   3. finalize (one CTA per sequence, a dependent launch): the exact top k
//      of each row's candidates, by rank counting.  If fewer than k logits
//      reached tau0, or more than the buffer holds, the row's top k is
//      recomputed exactly by re-scanning the row with a rising key threshold.
//      Then the temperature, the renormalisation over the top k and the top-p
//      cut, the accept tests, and the emitted token by an exponential race
//      over the few kept ids.
#include "spv_internal.h"
#include "spv_stream.cuh"

#include <climits>

#include "spv.h"

namespace spv {

constexpr int TOPK_MAX = 64;               // largest top_k
constexpr int CAND_CAP = 512;              // candidates of a row the finalize sorts (>= 8 k)
constexpr int CPB = 16;                    // candidate slots per 1024-logit block
constexpr uint32_t STREAM_FILTERED = 8;    // Philox stream of the filtered race
constexpr int SAMPLE_BLOCKS = 8;           // 1024-logit blocks sampled per row
constexpr int FALLBACK_ITERS = 64;         // re-scans of a row before giving up (bad row)

static_assert(SPV_MAX_TOP_K == TOPK_MAX, "top_k limit must match the API");

struct FiltParams {
    long long total_items;
    int nc, nb, V;
    unsigned *err;
    const unsigned char *target, *draft;
    const int32_t *tokens;
    const float *r;
    const uint64_t *keys;
    int B, gamma, R;        // R = 2 gamma + 1 rows per sequence
    int top_k;
    float top_p, invT;
    int32_t *accept_count, *out_tokens;
    float *out_pq, *out_Z;
    int32_t *row_status;
    float *tau;             // [B*R] sampled threshold
    int *rbad;              // [B*R] NaN or +inf seen
    int *bcnt;              // [B*R][nb] logits of each block at or above tau
    uint64_t *cand;         // [B*R][nb][CPB] their keys (the first CPB of a block)
};

// Key of logit x at id i: order-preserving logit bits, then the inverted id,
// so keys sort by logit descending, then id ascending; every key is > 0.
__device__ __forceinline__ uint64_t filt_key(float x, int i)
{
    return (static_cast<uint64_t>(float_key(x)) << 32) | static_cast<uint64_t>(0xFFFFFFFFu - static_cast<uint32_t>(i));
}

__device__ __forceinline__ float key_value(uint64_t k)
{
    const uint32_t u = static_cast<uint32_t>(k >> 32);
    return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}

__device__ __forceinline__ int key_id(uint64_t k) { return static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(k)); }

// Row `row` = b * R + rho of a call: target row rho <= gamma, else draft row rho - gamma - 1.
template <int DT> __device__ __forceinline__ const unsigned char *filt_row_ptr(const FiltParams &P, long long row)
{
    constexpr int EB = DType<DT>::BYTES;
    const int b = static_cast<int>(div_row(row, P.R)), rho = static_cast<int>(row - static_cast<long long>(b) * P.R);
    if (rho <= P.gamma)
        return P.target + (static_cast<size_t>(b) * (P.gamma + 1) + rho) * static_cast<size_t>(P.V) * EB;
    return P.draft + (static_cast<size_t>(b) * P.gamma + (rho - P.gamma - 1)) * static_cast<size_t>(P.V) * EB;
}

__device__ __forceinline__ uint64_t shfl_u64(uint64_t v, int src)
{
    const uint32_t lo = __shfl_sync(0xffffffffu, static_cast<uint32_t>(v), src);
    const uint32_t hi = __shfl_sync(0xffffffffu, static_cast<uint32_t>(v >> 32), src);
    return (static_cast<uint64_t>(hi) << 32) | lo;
}

__device__ __forceinline__ float warp_incl_scan(float v, int lane)
{
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    return v;
}

__device__ __forceinline__ int id_hash(int x) { return static_cast<int>((static_cast<uint32_t>(x) * 2654435761u) >> 25); }

// Descending bitonic sort of 32 S keys, element 32 s + lane in a[s].
template <int S>
__device__ __forceinline__ void bitonic_desc(uint64_t (&a)[S], int lane)
{
    constexpr int N = 32 * S;
#pragma unroll
    for (int kk = 2; kk <= N; kk <<= 1) {
#pragma unroll
        for (int j = kk >> 1; j > 0; j >>= 1) {
            if (j >= 32) {  // partner in another slot of the same lane
                const int js = j >> 5;
#pragma unroll
                for (int sl = 0; sl < S; ++sl) {
                    if (sl & js) continue;
                    const bool desc = ((32 * sl + lane) & kk) == 0;
                    const uint64_t x = a[sl], y = a[sl | js];
                    const uint64_t hi = x > y ? x : y, lo = x > y ? y : x;
                    a[sl] = desc ? hi : lo;
                    a[sl | js] = desc ? lo : hi;
                }
            } else {
                const bool lower = (lane & j) == 0;
#pragma unroll
                for (int sl = 0; sl < S; ++sl) {
                    const uint32_t olo = __shfl_xor_sync(0xffffffffu, static_cast<uint32_t>(a[sl]), j);
                    const uint32_t ohi = __shfl_xor_sync(0xffffffffu, static_cast<uint32_t>(a[sl] >> 32), j);
                    const uint64_t o = (static_cast<uint64_t>(ohi) << 32) | olo;
                    const bool desc = ((32 * sl + lane) & kk) == 0;
                    a[sl] = (lower == desc) ? (a[sl] > o ? a[sl] : o) : (a[sl] < o ? a[sl] : o);
                }
            }
        }
    }
}

// Entry i of the merge of two descending 64-key lists A and B (the first i
// entries of the union are a of A and i - a of B: merge-path co-rank).
__device__ __forceinline__ uint64_t merged_entry(const uint64_t *A, const uint64_t *B, int i)
{
    int lo = i > TOPK_MAX ? i - TOPK_MAX : 0, hi = i < TOPK_MAX ? i : TOPK_MAX;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1, j = i - mid;
        if (j > 0 && A[mid] > B[j - 1]) lo = mid + 1;
        else hi = mid;
    }
    const int a = lo, j = i - lo;
    if (a >= TOPK_MAX) return B[j];
    if (j >= TOPK_MAX) return A[a];
    return A[a] > B[j] ? A[a] : B[j];
}

// ------------------------------------------------------------------ 1. sample
// One CTA per row: warp j takes the j-th of SAMPLE_BLOCKS evenly spaced
// blocks (every block when the row has no more) and each lane its two
// largest logits there; then warp 0 takes the m-th largest of those by m
// rounds of a warp max.  m distinct logits of the row reach it; when the
// whole row was sampled m = k, so at least min(k, V) logits reach it (k <=
// 64).  Also clears the row's NaN / +inf flag.
template <int DT>
__global__ void __launch_bounds__(SAMPLE_BLOCKS * 32) filt_sample_kernel(const FiltParams P)
{
    __shared__ float sv[SAMPLE_BLOCKS][64];
    // The streaming grid may be scheduled now: its copies do not depend on
    // this grid; its consumers wait for it (griddepcontrol.wait).
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row = blockIdx.x;
    constexpr int EB = DType<DT>::BYTES;
    const unsigned char *rp = filt_row_ptr<DT>(P, row);
    const int ns = P.nb < SAMPLE_BLOCKS ? P.nb : SAMPLE_BLOCKS;
    float m1 = -INFINITY, m2 = -INFINITY;
    if (warp < ns) {
        const int beta = static_cast<int>(static_cast<long long>(warp) * P.nb / ns);
        const int valid = min(G, P.V - beta * G);
        float v[32];
        load_block_global<DT>(v, rp + static_cast<size_t>(beta) * G * EB, lane, valid);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            const float x = v[e];
            if (x > m1) {
                m2 = m1;
                m1 = x;
            } else if (x > m2) {
                m2 = x;
            }
        }
    }
    sv[warp][lane] = m1;
    sv[warp][32 + lane] = m2;
    __syncthreads();
    if (warp != 0) return;
    constexpr int NS = 2 * SAMPLE_BLOCKS;
    float gm[NS];
#pragma unroll
    for (int j = 0; j < SAMPLE_BLOCKS; ++j) {
        gm[2 * j] = sv[j][lane];
        gm[2 * j + 1] = sv[j][32 + lane];
    }
    // m: about 3.5 k logits of the row expected at or above the m-th largest sampled logit
    int m = P.top_k;
    if (ns < P.nb) {
        const long long sampled = static_cast<long long>(ns) * G;
        const long long mm = (7LL * P.top_k * sampled + 2LL * P.V - 1) / (2LL * P.V);
        m = static_cast<int>(mm < 1 ? 1 : (mm < P.top_k ? mm : P.top_k));
    }
    // The m-th largest: every lane's values as order-preserving bit patterns
    // (NaN as -inf), sorted descending in registers by a bitonic network;
    // then m rounds, each taking the warp's largest head (one redux) from the
    // first lane that holds it.  -inf is never taken: fewer than m finite
    // sampled logits leave t = -inf.
    constexpr uint32_t KEY_NEG_INF = 0x007fffffu;  // the pattern of -inf
    uint32_t key[NS];
#pragma unroll
    for (int j = 0; j < NS; ++j) {
        const uint32_t u = __float_as_uint(isnan(gm[j]) ? -INFINITY : gm[j]);
        key[j] = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    }
#pragma unroll
    for (int size = 2; size <= NS; size <<= 1)
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1)
#pragma unroll
            for (int i = 0; i < NS; ++i) {
                const int j = i ^ stride;
                if (j > i) {
                    const uint32_t hi = max(key[i], key[j]), lo = min(key[i], key[j]);
                    const bool desc = (i & size) == 0;
                    key[i] = desc ? hi : lo;
                    key[j] = desc ? lo : hi;
                }
            }
    float t = -INFINITY;
    for (int round = 0; round < m; ++round) {
        const uint32_t mx = __reduce_max_sync(0xffffffffu, key[0]);
        if (mx <= KEY_NEG_INF) {  // fewer than m finite sampled logits
            t = -INFINITY;
            break;
        }
        const bool mine = lane == __ffs(__ballot_sync(0xffffffffu, key[0] == mx)) - 1;
#pragma unroll
        for (int j = 0; j + 1 < NS; ++j) key[j] = mine ? key[j + 1] : key[j];
        key[NS - 1] = mine ? 0u : key[NS - 1];
        t = __uint_as_float((mx & 0x80000000u) ? (mx & 0x7fffffffu) : ~mx);
    }
    if (lane == 0) {
        P.tau[row] = t;
        P.rbad[row] = 0;
    }
}

// ------------------------------------------------------------------ 2. stream
// Streaming op: compare every logit with its row's tau0, record how many of
// each block reach it and the keys of the first CPB, flag NaN / +inf.
template <int DT> struct FiltOp {
    using Params = FiltParams;
    static constexpr int EB = DType<DT>::BYTES;
    static constexpr int CTAS_PER_SM = DT == 0 ? 3 : 4;
    static constexpr bool WAITS_PRIOR = true;  // tau0 and the cleared flags come from filt_sample_kernel

    __device__ static __forceinline__ const void *row_ptr(const Params &P, long long row)
    {
        return filt_row_ptr<DT>(P, row);
    }

    __device__ static __forceinline__ float at(const unsigned char *blk, int i)
    {
        if (DT == 0) return reinterpret_cast<const float *>(blk)[i];
        return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const unsigned short *>(blk)[i]) << 16);
    }

    __device__ static __forceinline__ void block_smem(const Params &P, long long row, int beta, const unsigned char *blk,
                                                      int valid, int lane)
    {
        if constexpr (DT == 1) {
            const float tau = __ldcg(&P.tau[row]);
            if (__bfloat162float(__float2bfloat16_rn(tau)) == tau) {  // tau is a bf16 value: compare packed
                scan_bf16(P, row, beta, blk, valid, lane, tau);
                return;
            }
        }
        float v[32];
        load_block_smem<DT>(v, blk, lane);
        mask_tail<DT>(v, valid, lane);
        scan(P, row, beta, v, blk, valid, lane);
    }

    // bf16, packed: the lane's maximum by bf16x2 max with NaN propagation and
    // the elements reaching tau by bf16x2 >= masks (word q holds elements
    // 2q and 2q + 1 of the lane, as in the float copy); otherwise as scan.
    __device__ static __forceinline__ void scan_bf16(const Params &P, long long row, int beta, const unsigned char *blk,
                                                     int valid, int lane, float tau)
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
        if (valid < G) {  // -inf past the row's end
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const int e0 = (q >> 2) * 256 + lane * 8 + 2 * (q & 3);
                if (e0 >= valid) w[q] = (w[q] & 0xffff0000u) | 0xff80u;
                if (e0 + 1 >= valid) w[q] = (w[q] & 0x0000ffffu) | 0xff800000u;
            }
        }
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(w);
        __nv_bfloat162 mx2[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) mx2[a] = __hmax2_nan(h[a], h[a + 8]);
#pragma unroll
        for (int a = 0; a < 4; ++a) mx2[a] = __hmax2_nan(mx2[a], mx2[a + 4]);
        mx2[0] = __hmax2_nan(__hmax2_nan(mx2[0], mx2[1]), __hmax2_nan(mx2[2], mx2[3]));
        const float mx = max_nan(__low2float(mx2[0]), __high2float(mx2[0]));
        const size_t slot = static_cast<size_t>(row) * P.nb + beta;
        const bool bad = !(mx < INFINITY);  // NaN or +inf in the lane's logits
        if (__any_sync(0xffffffffu, bad) && lane == 0) atomicExch(&P.rbad[row], 1);
        const bool hit = !bad && mx >= tau;
        if (!__any_sync(0xffffffffu, hit)) {
            if (lane == 0) P.bcnt[slot] = 0;
            return;
        }
        uint32_t mask = 0;
        if (hit) {
            const __nv_bfloat162 t2 = __float2bfloat162_rn(tau);
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const unsigned m2 = __hge2_mask(h[q], t2);
                mask |= ((m2 & 1u) | ((m2 >> 15) & 2u)) << (2 * q);
            }
            if (valid < G) {  // the -inf padding is no candidate, even for tau = -inf
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    if (lane_index<DT>(lane, e) >= valid) mask &= ~(1u << e);
            }
        }
        emit(P, slot, beta, blk, mask, lane);
    }

    __device__ static __forceinline__ void block(const Params &P, long long row, int beta, float v[32], int valid,
                                                 int lane)
    {
        scan(P, row, beta, v, filt_row_ptr<DT>(P, row) + static_cast<size_t>(beta) * G * EB, valid, lane);
    }

    // v: the lane's 32 logits (-inf past the row's end); blk: the block in
    // shared or global memory, re-read for the rare candidates.
    __device__ static __forceinline__ void scan(const Params &P, long long row, int beta, const float v[32],
                                                const unsigned char *blk, int valid, int lane)
    {
        const float tau = __ldcg(&P.tau[row]);
        float mx = v[0];
#pragma unroll
        for (int e = 1; e < 32; ++e) mx = max_nan(mx, v[e]);
        const size_t slot = static_cast<size_t>(row) * P.nb + beta;
        const bool bad = !(mx < INFINITY);  // NaN or +inf in the lane's logits
        if (__any_sync(0xffffffffu, bad) && lane == 0) atomicExch(&P.rbad[row], 1);
        const bool hit = !bad && mx >= tau;
        if (!__any_sync(0xffffffffu, hit)) {
            if (lane == 0) P.bcnt[slot] = 0;
            return;
        }
        uint32_t mask = 0;
        if (hit) {
#pragma unroll
            for (int e = 0; e < 32; ++e) mask |= (v[e] >= tau ? 1u : 0u) << e;
            if (valid < G) {
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    if (lane_index<DT>(lane, e) >= valid) mask &= ~(1u << e);
            }
        }
        emit(P, slot, beta, blk, mask, lane);
    }

    // The block's count of elements at or above tau and the keys of the first
    // CPB (lane order, then element order within the lane).
    __device__ static __forceinline__ void emit(const Params &P, size_t slot, int beta, const unsigned char *blk,
                                                uint32_t mask, int lane)
    {
        const int c = __popc(mask);
        int off = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, off, o);
            if (lane >= o) off += u;
        }
        if (lane == 31) P.bcnt[slot] = off;
        off -= c;
        uint64_t *dst = P.cand + slot * CPB;
        for (uint32_t m = mask; m && off < CPB; m &= m - 1u, ++off) {
            const int i = lane_index<DT>(lane, __ffs(m) - 1);
            dst[off] = filt_key(at(blk, i), beta * G + i);
        }
    }
};

// ------------------------------------------------------------------ 3. finalize
constexpr int FILT_ROWS_MAX = 2 * 32 + 1;  // 2 gamma + 1 rows at gamma = SPV_MAX_GAMMA

struct FiltSmem {
    int x[32];
    float rr[32];
    int n[FILT_ROWS_MAX];       // kept ids per row
    int hid[2 * TOPK_MAX];      // id -> q' hash of the rejected position's draft row
    float hq[2 * TOPK_MAX];
    int rcnt[4 * NCW];          // candidates gathered per row of the current group
    int rover[4 * NCW];         // a block of the row had more candidates than its slots
    int bad;
    uint64_t key;
};

// FW warps per CTA (while the sequences fit on the SMs at once: 32 for more
// than 16 rows per sequence, else 16; 8 otherwise).
template <int FW> struct FiltFin {
    using Params = FiltParams;
    using Smem = FiltSmem;
    static constexpr int FIN_WARPS = FW;
    static_assert(FW <= 4 * NCW, "row counters sized for 32 warps");
    // keys [rows][64] (u64), probs [rows][64], per-warp candidate staging
    static constexpr int KEYS_FLOATS = FILT_ROWS_MAX * TOPK_MAX * 2;
    static constexpr int PROBS_FLOATS = FILT_ROWS_MAX * TOPK_MAX;
    static constexpr int STAGE_FLOATS = FIN_WARPS * CAND_CAP * 2;
    static constexpr int HIST_FLOATS = FIN_WARPS * 256;
    static constexpr int FIN_BUF_FLOATS = KEYS_FLOATS + PROBS_FLOATS + STAGE_FLOATS + HIST_FLOATS;

    // Sort 64 keys (zeros pad) into out[0..64), descending; keep the first
    // `lim` (zeros after).  Register bitonic network.  Warp.
    __device__ static __forceinline__ void sort64(uint64_t a0, uint64_t a1, int lim, uint64_t *out, int lane)
    {
        uint64_t a[2] = {a0, a1};
        bitonic_desc<2>(a, lane);
        out[lane] = lane < lim ? a[0] : 0ull;
        out[32 + lane] = 32 + lane < lim ? a[1] : 0ull;
        __syncwarp();
    }

    // out[0..64): the largest min(k, c) of the c (<= CAND_CAP) distinct keys
    // in st, descending, zeros after.  More than 64 keys: a radix select on
    // the 32 logit bits of the keys (four 8-bit digits, most significant
    // first, counted in the warp's histogram `hist`) finds the logit of the
    // k-th largest key; the keys at or above it (k plus any ties) are then
    // sorted.  Warp; st is overwritten.
    __device__ static void sort_topk(uint64_t *st, int c, int k, uint64_t *out, int *hist, int lane)
    {
        const int lim = k < c ? k : c;
        if (c <= 64) {
            sort64(lane < c ? st[lane] : 0ull, 32 + lane < c ? st[32 + lane] : 0ull, lim, out, lane);
            return;
        }
        uint32_t prefix = 0u, pmask = 0u;
        int kr = k;  // rank sought among the keys matching the prefix
        for (int d = 3; d >= 0; --d) {
            const int sh = 8 * d;
#pragma unroll
            for (int h = 0; h < 8; ++h) hist[32 * h + lane] = 0;
            __syncwarp();
            for (int i = lane; i < c; i += 32) {
                const uint32_t k32 = static_cast<uint32_t>(st[i] >> 32);
                if ((k32 & pmask) == prefix) atomicAdd(&hist[(k32 >> sh) & 255u], 1);
            }
            __syncwarp();
            // lane l owns bins 255 - 8 l .. 248 - 8 l (descending)
            int cnt8[8], tot = 0;
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                cnt8[h] = hist[255 - 8 * lane - h];
                tot += cnt8[h];
            }
            int incl = tot;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += u;
            }
            const int before = incl - tot;  // keys in higher bins than this lane's
            int bin = -1, above = 0;
            if (before < kr && incl >= kr) {
                int run = before;
#pragma unroll
                for (int h = 0; h < 8; ++h) {
                    if (bin < 0 && run + cnt8[h] >= kr) {
                        bin = 255 - 8 * lane - h;
                        above = run;
                    }
                    run += cnt8[h];
                }
            }
            const unsigned who = __ballot_sync(0xffffffffu, bin >= 0);
            const int src = __ffs(who) - 1;
            bin = __shfl_sync(0xffffffffu, bin, src);
            above = __shfl_sync(0xffffffffu, above, src);
            prefix |= static_cast<uint32_t>(bin) << sh;
            pmask |= 255u << sh;
            kr -= above;
            __syncwarp();
        }
        // keys with logit bits >= prefix: the k-th largest and everything above
        int n = 0;
        const unsigned below = (1u << lane) - 1u;
        for (int i0 = 0; i0 < c; i0 += 32) {
            const int i = i0 + lane;
            const uint64_t key = i < c ? st[i] : 0ull;
            const bool take = i < c && static_cast<uint32_t>(key >> 32) >= prefix;
            const unsigned m = __ballot_sync(0xffffffffu, take);
            __syncwarp();
            if (take) st[n + __popc(m & below)] = key;  // n + rank <= i: compacting in place is safe
            n += __popc(m);
            __syncwarp();
        }
        if (n <= 64) {
            sort64(lane < n ? st[lane] : 0ull, 32 + lane < n ? st[32 + lane] : 0ull, lim, out, lane);
            return;
        }
        // many equal logits at the cut: sort the first 64 of them, merge in the rest 64 at a time
        sort64(st[lane], st[32 + lane], 64, out, lane);
        for (int j0 = 64; j0 < n; j0 += 64) {
            uint64_t a[2] = {j0 + lane < n ? st[j0 + lane] : 0ull, j0 + 32 + lane < n ? st[j0 + 32 + lane] : 0ull};
            bitonic_desc<2>(a, lane);
            __syncwarp();
            st[lane] = a[0];
            st[32 + lane] = a[1];
            __syncwarp();
            const uint64_t x = merged_entry(out, st, lane), y = merged_entry(out, st, 32 + lane);
            __syncwarp();
            out[lane] = x;
            out[32 + lane] = y;
            __syncwarp();
        }
        out[lane] = lane < lim ? out[lane] : 0ull;
        out[32 + lane] = 32 + lane < lim ? out[32 + lane] : 0ull;
        __syncwarp();
    }

    // The exact top k of a row whose candidates did not fit (or were too
    // few): re-scan the row keeping keys above a threshold -- from `thr`
    // (just below tau0's key when at least k logits reached tau0, else 0),
    // rising to just below the k-th largest kept key -- until at most
    // CAND_CAP remain.  Returns false if that took more than FALLBACK_ITERS
    // passes.
    template <int DT>
    __device__ static bool exact_rescan(const Params &P, long long row, uint64_t thr, uint64_t *st, uint64_t *out,
                                        int *hist, int lane)
    {
        const unsigned char *rp = filt_row_ptr<DT>(P, row);
        const unsigned below = (1u << lane) - 1u;
        for (int iter = 0; iter < FALLBACK_ITERS; ++iter) {
            int c = 0;
            for (int x0 = 0; x0 < P.V; x0 += 32) {
                const int x = x0 + lane;
                const float z = x < P.V ? DType<DT>::load(rp, x) : __int_as_float(0x7fffffff);
                const uint64_t K = z == z ? filt_key(z, x) : 0ull;
                const bool take = K > thr;
                const unsigned m = __ballot_sync(0xffffffffu, take);
                const int pos = c + __popc(m & below);
                if (take && pos < CAND_CAP) st[pos] = K;
                c += __popc(m);
            }
            __syncwarp();
            sort_topk(st, c < CAND_CAP ? c : CAND_CAP, P.top_k, out, hist, lane);
            if (c <= CAND_CAP) return true;
            thr = out[P.top_k - 1] - 1ull;  // c > CAND_CAP >= k: out holds k keys
            __syncwarp();
        }
        return false;
    }

    // Index of id x in a filtered row (-1 if not kept).  Whole warp, same x.
    __device__ static __forceinline__ int find(const uint64_t *keys, int n, int x, int lane)
    {
        const unsigned m0 = __ballot_sync(0xffffffffu, lane < n && key_id(keys[lane]) == x);
        const unsigned m1 = __ballot_sync(0xffffffffu, 32 + lane < n && key_id(keys[32 + lane]) == x);
        return m0 ? __ffs(m0) - 1 : (m1 ? 31 + __ffs(m1) : -1);
    }

    template <int DT>
    __device__ static void finalize_dt(const Params &P, int b, Smem &sm, float *buf, int warp, int lane)
    {
        const int g = P.gamma, R = P.R, K = P.top_k;
        uint64_t *keys = reinterpret_cast<uint64_t *>(buf);
        float *probs = buf + KEYS_FLOATS;
        uint64_t *stage = reinterpret_cast<uint64_t *>(buf + KEYS_FLOATS + PROBS_FLOATS);
        uint64_t *st = stage + warp * CAND_CAP;
        int *hist = reinterpret_cast<int *>(buf + KEYS_FLOATS + PROBS_FLOATS + STAGE_FLOATS) + warp * 256;
        // A. Inputs (before the dependent-grid wait).
        if (threadIdx.x == 0) {
            sm.bad = 0;
            sm.key = P.keys[b];
        }
        if (warp == 0 && lane < g) {
            sm.x[lane] = P.tokens[static_cast<size_t>(b) * g + lane];
            sm.rr[lane] = P.r[static_cast<size_t>(b) * g + lane];
        }
        asm volatile("griddepcontrol.wait;" ::: "memory");
        __syncthreads();
        if (warp == 0 && lane < g && (sm.x[lane] < 0 || sm.x[lane] >= P.V)) atomicOr(&sm.bad, 1);
        // B. Rows in groups of FW.  The whole CTA gathers the group's
        //    candidates from the blocks' slots into one staging row per warp
        //    (positions from a shared counter: the order does not matter, the
        //    warp sorts them), then one warp per row finds the exact top k
        //    and applies the filter.
        constexpr int NT = FW * 32;
        const int need = K < P.V ? K : P.V;
        for (int r0 = 0; r0 < R; r0 += FW) {
            const int nrows = R - r0 < FW ? R - r0 : FW;
            if (threadIdx.x < FW) {
                sm.rcnt[threadIdx.x] = 0;
                sm.rover[threadIdx.x] = 0;
            }
            __syncthreads();
            const int nslot = nrows * P.nb;
            for (int s0 = 0; s0 < nslot; s0 += 4 * NT) {
                int nbv[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int slot = s0 + u * NT + static_cast<int>(threadIdx.x);
                    nbv[u] = 0;
                    if (slot < nslot) {
                        const int rr = slot / P.nb;
                        nbv[u] = __ldcg(&P.bcnt[(static_cast<size_t>(b) * R + r0 + rr) * P.nb + (slot - rr * P.nb)]);
                    }
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int slot = s0 + u * NT + static_cast<int>(threadIdx.x);
                    if (slot < nslot && nbv[u] > 0) {
                        const int rr = slot / P.nb;
                        if (nbv[u] > CPB) {
                            sm.rover[rr] = 1;
                        } else {
                            const int pos = atomicAdd(&sm.rcnt[rr], nbv[u]);
                            uint64_t *dstw = stage + rr * CAND_CAP;
                            const uint64_t *src =
                                P.cand + ((static_cast<size_t>(b) * R + r0 + rr) * P.nb + (slot - rr * P.nb)) * CPB;
#pragma unroll
                            for (int t = 0; t < CPB; ++t)
                                if (t < nbv[u] && pos + t < CAND_CAP) dstw[pos + t] = __ldcg(&src[t]);
                        }
                    }
                }
            }
            __syncthreads();
            const int rho = r0 + warp;
            if (warp < nrows) {
                const long long row = static_cast<long long>(b) * R + rho;
                uint64_t *out = keys + rho * TOPK_MAX;
                bool bad = __ldcg(&P.rbad[row]) != 0;
                if (!bad) {
                    const int total = sm.rcnt[warp];
                    if (!sm.rover[warp] && total <= CAND_CAP && total >= need) {
                        sort_topk(st, total, K, out, hist, lane);
                    } else {
                        const float tau = __ldcg(&P.tau[row]);
                        const uint64_t thr = (total >= need && tau > -INFINITY)
                                                 ? (static_cast<uint64_t>(float_key(tau)) << 32) - 1ull : 0ull;
                        bad = !exact_rescan<DT>(P, row, thr, st, out, hist, lane);
                    }
                }
            const uint64_t lo = out[lane], hi = out[32 + lane];
            // Filter: renormalise over the top k, then the top-p prefix.
            const uint64_t k0 = shfl_u64(lo, 0);
            const float m = key_value(k0);
            bad |= (k0 == 0ull) || !(m > -INFINITY);
            const float ea = lo != 0ull ? expf((key_value(lo) - m) * P.invT) : 0.f;
            const float eb = hi != 0ull ? expf((key_value(hi) - m) * P.invT) : 0.f;
            const int nvalid = __popc(__ballot_sync(0xffffffffu, lo != 0ull)) + __popc(__ballot_sync(0xffffffffu, hi != 0ull));
            const float ca = warp_incl_scan(ea, lane);
            const float cb = __shfl_sync(0xffffffffu, ca, 31) + warp_incl_scan(eb, lane);
            const float S = __shfl_sync(0xffffffffu, cb, 31);
            int n = nvalid;
            float Sk = S;
            if (P.top_p < 1.f && nvalid > 0) {
                const float lim = P.top_p * S;
                const int below = __popc(__ballot_sync(0xffffffffu, lo != 0ull && ca < lim)) +
                                  __popc(__ballot_sync(0xffffffffu, hi != 0ull && cb < lim));
                n = min(below + 1, nvalid);
                const float sa = __shfl_sync(0xffffffffu, ca, (n - 1) & 31), sb = __shfl_sync(0xffffffffu, cb, (n - 1) & 31);
                Sk = n <= 32 ? sa : sb;
            }
            probs[rho * TOPK_MAX + lane] = lane < n ? ea / Sk : 0.f;
            probs[rho * TOPK_MAX + 32 + lane] = 32 + lane < n ? eb / Sk : 0.f;
                if (lane == 0) {
                    sm.n[rho] = n;
                    if (bad) atomicOr(&sm.bad, 1);
                }
            }
            __syncthreads();  // the staging rows are free again
        }
        if (warp != 0) return;
        if (sm.bad) {
            write_bad(P, b, lane);
            return;
        }
        // C. Accept tests (one warp-wide lookup per position), first rejection.
        bool accl = false;
        for (int i = 0; i < g; ++i) {
            const int x = sm.x[i], dr = g + 1 + i;
            const int jp = find(keys + i * TOPK_MAX, sm.n[i], x, lane);
            const int jq = find(keys + dr * TOPK_MAX, sm.n[dr], x, lane);
            const float p = jp >= 0 ? probs[i * TOPK_MAX + jp] : 0.f;
            const float q = jq >= 0 ? probs[dr * TOPK_MAX + jq] : 0.f;
            if (lane == i) accl = (p > 0.f) && (sm.rr[i] * q <= p);
            if (P.out_pq && lane == 0) {
                P.out_pq[(static_cast<size_t>(b) * g + i) * 2] = p;
                P.out_pq[(static_cast<size_t>(b) * g + i) * 2 + 1] = q;
            }
        }
        const unsigned mask = __ballot_sync(0xffffffffu, accl);
        const unsigned all = (g == 32) ? 0xffffffffu : ((1u << g) - 1u);
        const int k = ((mask & all) == all) ? g : (__ffs(~mask) - 1);
        // D. The emitted token: race over the kept ids of target row k with
        //    masses p' (bonus) or max(0, p' - q') (residual; q' from a hash of
        //    draft row k).
        if (k < g) {
            const int dr = g + 1 + k, nd = sm.n[dr];
#pragma unroll
            for (int h = 0; h < 4; ++h) sm.hid[32 * h + lane] = -1;
            __syncwarp();
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int j = lane + 32 * h;
                if (j < nd) {
                    const int id = key_id(keys[dr * TOPK_MAX + j]);
                    int slot = id_hash(id);
                    for (int t = 0; t < 2 * TOPK_MAX && atomicCAS(&sm.hid[slot], -1, id) != -1; ++t)
                        slot = (slot + 1) & (2 * TOPK_MAX - 1);
                    sm.hq[slot] = probs[dr * TOPK_MAX + j];
                }
            }
            __syncwarp();
        }
        const int n = sm.n[k];
        const uint64_t key = sm.key;
        float best = INFINITY, z = 0.f;
        int bid = INT_MAX;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int j = lane + 32 * h;
            if (j < n) {
                const int id = key_id(keys[k * TOPK_MAX + j]);
                float w = probs[k * TOPK_MAX + j];
                if (k < g) {
                    int slot = id_hash(id);
                    float q = 0.f;
                    for (int t = 0; t < 2 * TOPK_MAX; ++t) {
                        const int hv = sm.hid[slot];
                        if (hv == id) {
                            q = sm.hq[slot];
                            break;
                        }
                        if (hv == -1) break;
                        slot = (slot + 1) & (2 * TOPK_MAX - 1);
                    }
                    w = fmaxf(__fsub_rn(w, q), 0.f);
                }
                z += w;
                if (w > 0.f) {
                    uint32_t wd[4];
                    philox_group(wd, key, STREAM_FILTERED, 0u, static_cast<uint32_t>(id) >> 2);
                    const float A = arrival(expo(wd[id & 3]), 1.f / w);
                    if (A < best || (A == best && id < bid)) {
                        best = A;
                        bid = id;
                    }
                }
            }
        }
        warp_argmin(best, bid);
        z = warp_sum(z);
        if (bid == INT_MAX) {  // no mass to draw from: bad row
            write_bad(P, b, lane);
            return;
        }
        for (int i = lane; i <= g; i += 32) {
            int v = -1;
            if (i < k) v = sm.x[i];
            else if (i == k) v = bid;
            P.out_tokens[static_cast<size_t>(b) * (g + 1) + i] = v;
        }
        if (lane == 0) {
            P.accept_count[b] = k;
            if (P.row_status) P.row_status[b] = 0;
            if (P.out_Z) P.out_Z[b] = (k == g) ? 1.f : z;
        }
    }

    __device__ static void write_bad(const Params &P, int b, int lane)
    {
        const int g = P.gamma;
        for (int i = lane; i <= g; i += 32) P.out_tokens[static_cast<size_t>(b) * (g + 1) + i] = -1;
        if (P.out_pq)
            for (int i = lane; i < 2 * g; i += 32) P.out_pq[static_cast<size_t>(b) * 2 * g + i] = __int_as_float(0x7fffffff);
        if (lane == 0) {
            P.accept_count[b] = -1;
            if (P.row_status) P.row_status[b] = STATUS_BAD_ROW;
            if (P.out_Z) P.out_Z[b] = __int_as_float(0x7fffffff);
        }
    }
};

// The finalize of one dtype (finalize_kernel calls Fin::finalize).
template <int DT, int FW> struct FiltFinDT : FiltFin<FW> {
    using Base = FiltFin<FW>;
    __device__ static void finalize(const typename Base::Params &P, int b, typename Base::Smem &sm, float *buf, int warp,
                                    int lane)
    {
        Base::template finalize_dt<DT>(P, b, sm, buf, warp, lane);
    }
};

// ------------------------------------------------------------------ host launch
size_t filtered_ws_bytes(int B, int gamma, int V)
{
    const size_t rows = static_cast<size_t>(B) * (2 * static_cast<size_t>(gamma) + 1), nb = blocks_per_row(V);
    size_t n = WS_HEADER;
    n += align256(rows * 4) * 2;              // tau, rbad
    n += align256(rows * nb * 4);             // per-block candidate counts
    n += align256(rows * nb * CPB * 8);       // candidate keys
    const size_t gr = greedy_ws_bytes(B, gamma, V);
    return n > gr ? n : gr;
}

template <int DT>
static cudaError_t launch_filtered_dt(const FiltParams &P, bool tma, cudaStream_t st)
{
    const long long rows = static_cast<long long>(P.B) * P.R;
    filt_sample_kernel<DT><<<static_cast<unsigned>(rows), SAMPLE_BLOCKS * 32, 0, st>>>(P);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    int sms = 0;
    if ((e = device_sm_count(&sms)) != cudaSuccess) return e;
    // One finalize CTA per sequence: 16 warps while the sequences fit on the
    // SMs at once, else 8 (two CTAs per SM).
    // More than 16 rows per sequence (gamma >= 8): 32 warps select every
    // row's top k at once (64 registers, 214 KB of shared memory) instead of
    // two groups of 16 in turn (eagle gamma = 15, B = 32: 85.3 -> 79.5 us).
    if (P.B <= sms && P.R > 16) return launch_stream_finalize<FiltOp<DT>, FiltFinDT<DT, 32>, DT>(P, tma, P.B, st);
    return P.B <= sms ? launch_stream_finalize<FiltOp<DT>, FiltFinDT<DT, 16>, DT>(P, tma, P.B, st)
                      : launch_stream_finalize<FiltOp<DT>, FiltFinDT<DT, NCW>, DT>(P, tma, P.B, st);
}

cudaError_t launch_filtered(const ChainLaunch &L, cudaStream_t st)
{
    FiltParams P{};
    P.V = L.V;
    P.nb = blocks_per_row(L.V);
    P.nc = chunks_per_row(L.V);
    P.B = L.B;
    P.gamma = L.gamma;
    P.R = 2 * L.gamma + 1;
    P.total_items = static_cast<long long>(L.B) * P.R * P.nc;
    const size_t rows = static_cast<size_t>(L.B) * P.R;
    unsigned char *ws = static_cast<unsigned char *>(L.ws);
    P.err = reinterpret_cast<unsigned *>(ws);
    size_t off = WS_HEADER;
    P.tau = reinterpret_cast<float *>(ws + off);
    off += align256(rows * 4);
    P.rbad = reinterpret_cast<int *>(ws + off);
    off += align256(rows * 4);
    P.bcnt = reinterpret_cast<int *>(ws + off);
    off += align256(rows * P.nb * 4);
    P.cand = reinterpret_cast<uint64_t *>(ws + off);
    P.target = static_cast<const unsigned char *>(L.target);
    P.draft = static_cast<const unsigned char *>(L.draft);
    P.tokens = L.tokens;
    P.r = L.r;
    P.keys = L.keys;
    P.top_k = L.top_k;
    P.top_p = L.top_p;
    P.invT = 1.0f / L.T;
    P.accept_count = L.accept_count;
    P.out_tokens = L.out_tokens;
    P.out_pq = L.out_pq;
    P.out_Z = L.out_Z;
    P.row_status = L.row_status;
    return L.dtype == 0 ? launch_filtered_dt<0>(P, L.tma, st) : launch_filtered_dt<1>(P, L.tma, st);
}

}  // namespace spv
