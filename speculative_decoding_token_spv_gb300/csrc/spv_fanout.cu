// spv_fanout.cu -- top-F_k bonus-candidate fan-out over draft logits.
//
// "Speculative Speculative Decoding" (review of arXiv 2603.03251), Figure 2:
// at each position k the speculation cache takes F_k bonus-token candidates
// from the top ranks of the draft logits, excluding the token already sent for
// verification.  Keys are 64-bit (order-preserving logit key, inverted id), so
// logit descending then id ascending, every key distinct.  One pass over the
// rows: each warp reduces a 1024-logit block to its own sorted top-F list (the
// F-th largest lane maximum bounds the block's F-th largest key from below;
// the elements that reach it are ranked or sorted once); the finalize grid
// (one CTA per row) merges the per-block lists into the row's top-F, by the
// same kind of bound over the list heads when the lists fit in shared memory,
// else list by list.
#include "spv_internal.h"
#include "spv_stream.cuh"

namespace spv {

constexpr int FAN_MAX_LISTS_PER_LANE = 4;  // blocks per row <= 8 warps * 32 lanes * 4

struct FanoutParams {
    long long total_items;
    int nc, nb, V;
    unsigned *err;
    const unsigned char *draft;
    const int32_t *exclude;
    int K1, Fmax, sumF;
    int F[64];
    int off[65];
    int32_t *out_ids, *row_status;
    uint64_t *cand;  // [rows*nb*Fmax]; UINT64_MAX in slot 0 marks a NaN block, 0 = no candidate
};

constexpr int FAN_CACHE = 4096;  // candidates staged in shared memory when nb * F fits

struct FanoutSmem {
    uint64_t cand[FAN_CACHE];
    uint64_t list[NCW][64];
    int bad;
    int fast;  // the row's ids were written by the threshold merge
};

__device__ __forceinline__ uint64_t cand_key(uint32_t k32, int id)
{
    return (static_cast<uint64_t>(k32) << 32) | static_cast<uint64_t>(0xFFFFFFFFu - static_cast<uint32_t>(id));
}

// Id of a candidate key (0 = no candidate: -1).
__device__ __forceinline__ int32_t cand_id(uint64_t key)
{
    return key ? static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(key)) : -1;
}

// Rank of the key a among the keys held by lanes 0..n-1 (one per lane,
// distinct): the number of larger ones, i.e. its position in descending order.
__device__ __forceinline__ int rank_desc(uint64_t a, int n)
{
    int rank = 0;
    for (int j = 0; j < n; ++j) rank += __shfl_sync(0xffffffffu, a, j) > a ? 1 : 0;
    return rank;
}

// Descending bitonic sort of 64 keys held two per lane (element i = lane in
// a, element i = lane + 32 in c); afterwards a holds rank lane, c rank lane + 32.
__device__ __forceinline__ void bitonic64_desc(uint64_t &a, uint64_t &c, int lane)
{
#pragma unroll
    for (int kk = 2; kk <= 64; kk <<= 1) {
#pragma unroll
        for (int j = kk >> 1; j > 0; j >>= 1) {
            if (j == 32) {
                // partner of i is i + 32 (same lane): i = lane < 32 is the lower one
                const bool desc = (lane & kk) == 0;  // kk == 64: whole sequence descending
                const uint64_t hi = a > c ? a : c, lo = a > c ? c : a;
                a = desc ? hi : lo;
                c = desc ? lo : hi;
            } else {
                const uint64_t oa = __shfl_xor_sync(0xffffffffu, a, j);
                const uint64_t oc = __shfl_xor_sync(0xffffffffu, c, j);
                const bool lower = (lane & j) == 0;
                const bool da = ((lane & kk) == 0), dc = (((lane + 32) & kk) == 0);
                a = (lower == da) ? (a > oa ? a : oa) : (a < oa ? a : oa);
                c = (lower == dc) ? (c > oc ? c : oc) : (c < oc ? c : oc);
            }
        }
    }
}

template <int DT> struct FanoutOp {
    using Params = FanoutParams;
    using Smem = FanoutSmem;
    static constexpr int EB = DType<DT>::BYTES;

    __device__ static __forceinline__ const void *row_ptr(const Params &P, long long row)
    {
        return P.draft + static_cast<size_t>(row) * static_cast<size_t>(P.V) * EB;
    }

    static constexpr int CTAS_PER_SM = 3;

    // Key of element e of the lane from the staged block (the same element
    // lane_index(lane, e) as in the register copy); 0 = not a candidate.
    __device__ static __forceinline__ uint32_t smem_key(const unsigned char *blk, int lane, int e, int valid, int base,
                                                        int ex)
    {
        const int i = lane_index<DT>(lane, e);
        float x;
        if (DT == 0) x = reinterpret_cast<const float *>(blk)[i];
        else x = __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const unsigned short *>(blk)[i]) << 16);
        return (i < valid && base + i != ex && x == x) ? float_key(x) : 0u;
    }

    // Top-F of a block staged in shared memory.  The F-th largest of the 32
    // lane maxima bounds the block's F-th largest key from below (F distinct
    // elements reach it), so only elements at or above it can be in the
    // top F (keys re-read from the staged block).  F > 32 visits every
    // element.
    __device__ static __forceinline__ void block_smem(const Params &P, long long row, int beta,
                                                      const unsigned char *blk, int valid, int lane)
    {
        const int k = static_cast<int>(row - div_row(row, P.K1) * P.K1);
        const int F = P.F[k];
        if (F == 0) return;
        const int ex = P.exclude[row];
        const int base = beta * G;
        float v[32];
        load_block_smem<DT>(v, blk, lane);
        uint64_t *out = P.cand + (static_cast<size_t>(row) * P.nb + beta) * P.Fmax;
        uint32_t mask = 0;
        if (valid == G && !(ex >= base && ex < base + G)) {
            // A full block without the excluded id: every element is a
            // candidate unless NaN (then the row is bad).  Lane maximum by
            // max.NaN, the threshold among the lane maxima as floats (the
            // order of the keys), then one compare per element.
            float m8[8];
#pragma unroll
            for (int a = 0; a < 8; ++a) m8[a] = max_nan(max_nan(v[a], v[a + 8]), max_nan(v[a + 16], v[a + 24]));
            const float mx = max_nan(max_nan(max_nan(m8[0], m8[1]), max_nan(m8[2], m8[3])),
                                     max_nan(max_nan(m8[4], m8[5]), max_nan(m8[6], m8[7])));
            if (__any_sync(0xffffffffu, mx != mx)) {
                if (lane == 0) out[0] = ~0ull;
                return;
            }
            if (F <= 32) {
                float sv = mx;
#pragma unroll
                for (int kk = 2; kk <= 32; kk <<= 1) {
#pragma unroll
                    for (int j = kk >> 1; j > 0; j >>= 1) {
                        const float o = __shfl_xor_sync(0xffffffffu, sv, j);
                        const bool desc = (lane & kk) == 0, lower = (lane & j) == 0;
                        sv = (lower == desc) ? fmaxf(sv, o) : fminf(sv, o);
                    }
                }
                const float t = __shfl_sync(0xffffffffu, sv, F - 1);
#pragma unroll
                for (int e = 0; e < 32; ++e) mask |= (v[e] >= t ? 1u : 0u) << e;
            } else {
                mask = 0xffffffffu;
            }
            select_top(P, row, beta, blk, valid, lane, ex, F, mask, out);
            return;
        }
        general_block(P, row, beta, blk, valid, lane, ex, F, out);
    }

    // The ragged tail block or the block holding the excluded id: keys with
    // 0 for the elements that are not candidates (out of line: it runs at
    // most twice per row and keeps its registers out of the fast path).
    __device__ __noinline__ static void general_block(const Params &P, long long row, int beta,
                                                      const unsigned char *blk, int valid, int lane, int ex, int F,
                                                      uint64_t *out)
    {
        const int base = beta * G;
        float v[32];
        load_block_smem<DT>(v, blk, lane);
        uint32_t mask = 0;
        uint32_t key[32];
        bool nan = false;
        uint32_t lmax = 0;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            const int i = lane_index<DT>(lane, e);
            const float x = v[e];
            nan |= (x != x) && i < valid;
            key[e] = (i < valid && base + i != ex && x == x) ? float_key(x) : 0u;
            lmax = key[e] > lmax ? key[e] : lmax;
        }
        nan = __any_sync(0xffffffffu, nan);
        if (nan) {
            if (lane == 0) out[0] = ~0ull;
            return;
        }
        uint32_t thr = 1u;  // keys of candidates are >= 1
        if (F <= 32) {
            // descending bitonic sort of the lane maxima across the warp
            uint32_t sv = lmax;
#pragma unroll
            for (int kk = 2; kk <= 32; kk <<= 1) {
#pragma unroll
                for (int j = kk >> 1; j > 0; j >>= 1) {
                    const uint32_t o = __shfl_xor_sync(0xffffffffu, sv, j);
                    const bool desc = (lane & kk) == 0, lower = (lane & j) == 0;
                    sv = (lower == desc) ? (sv > o ? sv : o) : (sv < o ? sv : o);
                }
            }
            const uint32_t t = __shfl_sync(0xffffffffu, sv, F - 1);
            thr = t > 1u ? t : 1u;
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) mask |= (key[e] >= thr ? 1u : 0u) << e;
        select_top(P, row, beta, blk, valid, lane, ex, F, mask, out);
    }

    // The block's top F among the candidates in mask (keys re-read from the
    // staged block).  Usually few elements reach the threshold: compact them
    // (<= 64) into the warp's shared slots, sort the 64-bit keys once
    // (bitonic, two per lane, descending) and keep the first F.  Otherwise F
    // rounds of a warp max over the candidates.
    __device__ static __forceinline__ void select_top(const Params &P, long long row, int beta,
                                                      const unsigned char *blk, int valid, int lane, int ex, int F,
                                                      uint32_t mask, uint64_t *out)
    {
        const int base = beta * G;
        __shared__ uint64_t slots[NCW][64];
        const int n = __popc(mask);
        int pre = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, pre, o);
            if (lane >= o) pre += y;
        }
        const int total = __shfl_sync(0xffffffffu, pre, 31);
        if (F <= 32 && total <= 64) {
            const int warp = threadIdx.x >> 5;
            uint64_t *sl = slots[warp];
            int pos = pre - n;
            for (uint32_t m = mask; m; m &= m - 1) {
                const int e = __ffs(m) - 1;
                sl[pos++] = cand_key(smem_key(blk, lane, e, valid, base, ex), base + lane_index<DT>(lane, e));
            }
            __syncwarp();
            uint64_t a = lane < total ? sl[lane] : 0ull, c = lane + 32 < total ? sl[lane + 32] : 0ull;
            __syncwarp();
            if (total <= 32) {
                // One key per lane: its rank is the number of larger keys
                // (keys are distinct), which is its position in the list.
                const int rk = rank_desc(a, total);
                if (lane < total && rk < F) out[rk] = a;
                if (lane >= total && lane < F) out[lane] = 0ull;
                return;
            }
            bitonic64_desc(a, c, lane);
            if (lane < F) out[lane] = a;
            return;
        }
        uint64_t prev = ~0ull;
        for (int t = 0; t < F; ++t) {
            uint64_t best = 0;
            for (uint32_t m = mask; m; m &= m - 1) {
                const int e = __ffs(m) - 1;
                const uint64_t K = cand_key(smem_key(blk, lane, e, valid, base, ex), base + lane_index<DT>(lane, e));
                if (K < prev && K > best) best = K;
            }
            best = warp_max_u64(best);
            if (lane == 0) out[t] = best;
            prev = best;
        }
    }

    __device__ static __forceinline__ void block(const Params &P, long long row, int beta, float v[32], int valid,
                                                 int lane)
    {
        const int k = static_cast<int>(row - div_row(row, P.K1) * P.K1);
        const int F = P.F[k];
        if (F == 0) return;
        const int ex = P.exclude[row];
        uint32_t key[32];
        bool nan = false;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            const int i = lane_index<DT>(lane, e);
            const float x = v[e];
            nan |= (x != x);
            key[e] = (i < valid && beta * G + i != ex && x == x) ? float_key(x) : 0u;
        }
        nan = __any_sync(0xffffffffu, nan);
        uint64_t *out = P.cand + (static_cast<size_t>(row) * P.nb + beta) * P.Fmax;
        if (nan) {
            if (lane == 0) out[0] = ~0ull;
            return;
        }
        uint64_t prev = ~0ull;
        for (int t = 0; t < F; ++t) {
            uint64_t best = 0;
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                if (key[e]) {
                    const uint64_t K = cand_key(key[e], beta * G + lane_index<DT>(lane, e));
                    if (K < prev && K > best) best = K;
                }
            }
            best = warp_max_u64(best);
            if (lane == 0) out[t] = best;
            prev = best;
        }
    }

    static constexpr int FIN_WARPS = NCW;
    static constexpr int FIN_BUF_FLOATS = 0;

    __device__ static void finalize(const Params &P, int row, Smem &sm, float *, int warp, int lane)
    {
        const int k = row % P.K1, b = row / P.K1;
        const int F = P.F[k];
        const int nb = P.nb;
        if (threadIdx.x == 0) {
            sm.bad = 0;
            sm.fast = 0;
        }
        asm volatile("griddepcontrol.wait;" ::: "memory");
        consumer_sync();
        const uint64_t *rc = P.cand + static_cast<size_t>(row) * nb * P.Fmax;
        const bool cached = nb * F <= FAN_CACHE;
        if (F > 0) {
            if (cached) {
                // stage every candidate (list beta, rank t) at cand[beta * F + t]
                for (int i0 = 0; i0 < nb * F; i0 += NCW * 32 * 4) {
                    uint64_t v[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int i = i0 + u * NCW * 32 + threadIdx.x;
                        v[u] = i < nb * F ? __ldcg(rc + static_cast<size_t>(i / F) * P.Fmax + (i % F)) : 0ull;
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int i = i0 + u * NCW * 32 + threadIdx.x;
                        if (i < nb * F) {
                            sm.cand[i] = v[u];
                            if (i % F == 0 && v[u] == ~0ull) sm.bad = 1;
                        }
                    }
                }
            } else {
                for (int beta = threadIdx.x; beta < nb; beta += NCW * 32)
                    if (__ldcg(rc + static_cast<size_t>(beta) * P.Fmax) == ~0ull) sm.bad = 1;
            }
        }
        consumer_sync();
        int32_t *ids = P.out_ids + static_cast<size_t>(b) * P.sumF + P.off[k];
        if (F == 0 || sm.bad) {
            for (int t = threadIdx.x; t < F; t += NCW * 32) ids[t] = -1;
            if (threadIdx.x == 0 && P.row_status) P.row_status[row] = (F > 0 && sm.bad) ? STATUS_BAD_ROW : 0;
            return;
        }
        if (cached && F <= 32) {
            // Threshold merge (one warp): the F-th largest of the lane maxima
            // of the list heads bounds the row's F-th largest key from below
            // (F distinct keys reach it), so only entries at or above it can
            // be in the top F; the lists are sorted, so each is scanned only
            // down to it.  Up to 64 such entries are sorted once; more fall
            // through to the level-by-level merge below.
            if (warp == 0) {
                uint64_t lm = 0;
                for (int beta = lane; beta < nb; beta += 32) {
                    const uint64_t h = sm.cand[beta * F];
                    lm = h > lm ? h : lm;
                }
                const int rk = rank_desc(lm, 32);  // nonzero lane maxima are distinct
                const unsigned sel = __ballot_sync(0xffffffffu, lm != 0ull && rk == F - 1);
                const uint64_t t = sel ? __shfl_sync(0xffffffffu, lm, __ffs(sel) - 1) : 1ull;
                int n = 0;
                for (int beta = lane; beta < nb; beta += 32)
                    for (int j = 0; j < F && sm.cand[beta * F + j] >= t; ++j) ++n;
                int pre = n;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, pre, o);
                    if (lane >= o) pre += y;
                }
                const int total = __shfl_sync(0xffffffffu, pre, 31);
                if (total <= 64) {
                    uint64_t *sl = sm.list[0];
                    int pos = pre - n;
                    for (int beta = lane; beta < nb; beta += 32)
                        for (int j = 0; j < F && sm.cand[beta * F + j] >= t; ++j) sl[pos++] = sm.cand[beta * F + j];
                    __syncwarp();
                    uint64_t a = lane < total ? sl[lane] : 0ull, c = lane + 32 < total ? sl[lane + 32] : 0ull;
                    if (total <= 32) {
                        const int r = rank_desc(a, total);
                        if (lane < total && r < F) ids[r] = cand_id(a);
                        if (lane >= total && lane < F) ids[lane] = -1;
                    } else {
                        bitonic64_desc(a, c, lane);
                        if (lane < F) ids[lane] = cand_id(a);
                    }
                    if (lane == 0) {
                        sm.fast = 1;
                        if (P.row_status) P.row_status[row] = 0;
                    }
                }
            }
            consumer_sync();
            if (sm.fast) return;
        }
        // Level 1: warp w merges the sorted lists of blocks beta = w + NCW * j.
        auto cand_at = [&](int beta, int t) -> uint64_t {
            return cached ? sm.cand[beta * F + t] : __ldcg(rc + static_cast<size_t>(beta) * P.Fmax + t);
        };
        int head[FAN_MAX_LISTS_PER_LANE];
        uint64_t cur[FAN_MAX_LISTS_PER_LANE];
#pragma unroll
        for (int q = 0; q < FAN_MAX_LISTS_PER_LANE; ++q) {
            const int beta = warp + NCW * (lane + 32 * q);
            head[q] = 0;
            cur[q] = beta < nb ? cand_at(beta, 0) : 0ull;
        }
        for (int t = 0; t < F; ++t) {
            uint64_t mine = 0;
#pragma unroll
            for (int q = 0; q < FAN_MAX_LISTS_PER_LANE; ++q) mine = cur[q] > mine ? cur[q] : mine;
            const uint64_t best = warp_max_u64(mine);
            if (best != 0 && mine == best) {
#pragma unroll
                for (int q = 0; q < FAN_MAX_LISTS_PER_LANE; ++q) {
                    if (cur[q] == best) {
                        const int beta = warp + NCW * (lane + 32 * q);
                        ++head[q];
                        cur[q] = head[q] < F ? cand_at(beta, head[q]) : 0ull;
                    }
                }
            }
            if (lane == 0) sm.list[warp][t] = best;
        }
        consumer_sync();
        // Level 2: warp 0 merges the NCW warp lists.
        if (warp == 0) {
            int h = 0;
            uint64_t c = lane < NCW ? sm.list[lane][0] : 0ull;
            for (int t = 0; t < F; ++t) {
                const uint64_t best = warp_max_u64(c);
                if (best != 0 && c == best) {
                    ++h;
                    c = h < F ? sm.list[lane][h] : 0ull;
                }
                if (lane == 0) ids[t] = cand_id(best);
            }
            if (lane == 0 && P.row_status) P.row_status[row] = 0;
        }
    }
};

size_t fanout_ws_bytes(int B, int K1, int V, int Fmax)
{
    const size_t rows = static_cast<size_t>(B) * K1, nb = blocks_per_row(V);
    const size_t f = Fmax > 0 ? static_cast<size_t>(Fmax) : 1;
    return WS_HEADER + align256(rows * nb * f * 8);
}

cudaError_t launch_fanout(const FanoutLaunch &L, cudaStream_t st)
{
    FanoutParams P{};
    P.V = L.V;
    P.nb = blocks_per_row(L.V);
    P.nc = chunks_per_row(L.V);
    P.K1 = L.K1;
    P.Fmax = L.Fmax > 0 ? L.Fmax : 1;
    P.sumF = L.off[L.K1];
    for (int i = 0; i < 64; ++i) P.F[i] = i < L.K1 ? L.F[i] : 0;
    for (int i = 0; i <= 64; ++i) P.off[i] = i <= L.K1 ? L.off[i] : L.off[L.K1];
    P.total_items = static_cast<long long>(L.B) * L.K1 * P.nc;
    unsigned char *ws = static_cast<unsigned char *>(L.ws);
    P.err = reinterpret_cast<unsigned *>(ws);
    P.cand = reinterpret_cast<uint64_t *>(ws + WS_HEADER);
    P.draft = static_cast<const unsigned char *>(L.draft);
    P.exclude = L.exclude;
    P.out_ids = L.out_ids;
    P.row_status = L.row_status;
    const int rows = L.B * L.K1;
    return L.dtype == 0 ? launch_stream_finalize<FanoutOp<0>, FanoutOp<0>, 0>(P, L.tma, rows, st)
                        : launch_stream_finalize<FanoutOp<1>, FanoutOp<1>, 1>(P, L.tma, rows, st);
}

}  // namespace spv
