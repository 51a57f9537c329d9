// spv_fanout.cu -- top-F_k bonus-candidate fan-out over draft logits.
//
// "Speculative Speculative Decoding" (review of arXiv 2603.03251), Figure 2:
// at each position k the speculation cache takes F_k bonus-token candidates
// from the top ranks of the draft logits, excluding the token already sent for
// verification.  One pass over the rows: each warp reduces a 1024-logit block
// to its own top-F list (F rounds of a warp max over 64-bit keys
// (order-preserving logit key, inverted id), so logit descending then id
// ascending, every key distinct); the CTA that finishes a row's last item
// merges the per-block lists (which are already sorted) into the row's top-F.
#include "spv_internal.h"
#include "spv_stream.cuh"

namespace spv {

constexpr int FAN_MAX_LISTS_PER_LANE = 4;  // blocks per row <= 8 warps * 32 lanes * 4

struct FanoutParams {
    long long total_items;
    int nc, nb, V;
    unsigned *counter;
    unsigned *err;
    const unsigned char *draft;
    const int32_t *exclude;
    int K1, Fmax, sumF;
    int F[64];
    int off[65];
    int32_t *out_ids, *row_status;
    uint64_t *cand;  // [rows*nb*Fmax]; UINT64_MAX in slot 0 marks a NaN block, 0 = no candidate
};

struct FanoutSmem {
    uint64_t list[NCW][64];
    int bad;
};

__device__ __forceinline__ uint64_t cand_key(uint32_t k32, int id)
{
    return (static_cast<uint64_t>(k32) << 32) | static_cast<uint64_t>(0xFFFFFFFFu - static_cast<uint32_t>(id));
}

template <int DT> struct FanoutOp {
    using Params = FanoutParams;
    using Smem = FanoutSmem;
    static constexpr int EB = DType<DT>::BYTES;

    __device__ static __forceinline__ const void *row_ptr(const Params &P, long long row)
    {
        return P.draft + static_cast<size_t>(row) * static_cast<size_t>(P.V) * EB;
    }
    __device__ static __forceinline__ int group(const Params &, long long row) { return static_cast<int>(row); }
    __device__ static __forceinline__ int items_per_group(const Params &P) { return P.nc; }

    __device__ static __forceinline__ void block(const Params &P, long long row, int beta, float v[32], int valid,
                                                 int lane)
    {
        const int k = static_cast<int>(row % P.K1);
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

    __device__ static void finalize(const Params &P, int row, Smem &sm, int warp, int lane)
    {
        const int k = row % P.K1, b = row / P.K1;
        const int F = P.F[k];
        if (threadIdx.x == 0) sm.bad = 0;
        consumer_sync();
        const uint64_t *rc = P.cand + static_cast<size_t>(row) * P.nb * P.Fmax;
        if (F > 0) {
            for (int beta = threadIdx.x; beta < P.nb; beta += NCW * 32)
                if (__ldcg(rc + static_cast<size_t>(beta) * P.Fmax) == ~0ull) sm.bad = 1;
        }
        consumer_sync();
        int32_t *ids = P.out_ids + static_cast<size_t>(b) * P.sumF + P.off[k];
        if (F == 0 || sm.bad) {
            for (int t = threadIdx.x; t < F; t += NCW * 32) ids[t] = -1;
            if (threadIdx.x == 0) {
                if (P.row_status) P.row_status[row] = (F > 0 && sm.bad) ? STATUS_BAD_ROW : 0;
                P.counter[row] = 0u;
            }
            consumer_sync();
            return;
        }
        // Level 1: warp w merges the sorted lists of blocks beta = w + NCW * j.
        int head[FAN_MAX_LISTS_PER_LANE];
        uint64_t cur[FAN_MAX_LISTS_PER_LANE];
#pragma unroll
        for (int q = 0; q < FAN_MAX_LISTS_PER_LANE; ++q) {
            const int beta = warp + NCW * (lane + 32 * q);
            head[q] = 0;
            cur[q] = beta < P.nb ? __ldcg(rc + static_cast<size_t>(beta) * P.Fmax) : 0ull;
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
                        cur[q] = head[q] < F ? __ldcg(rc + static_cast<size_t>(beta) * P.Fmax + head[q]) : 0ull;
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
                if (lane == 0) ids[t] = best ? static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(best)) : -1;
            }
            if (lane == 0) {
                if (P.row_status) P.row_status[row] = 0;
                P.counter[row] = 0u;
            }
        }
        consumer_sync();
    }
};

template <class Op, int DT> static cudaError_t launch_fan(const typename Op::Params &P, bool tma, cudaStream_t st)
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

size_t fanout_ws_bytes(int B, int K1, int V, int Fmax)
{
    const size_t rows = static_cast<size_t>(B) * K1, nb = blocks_per_row(V);
    const size_t f = Fmax > 0 ? static_cast<size_t>(Fmax) : 1;
    return WS_HEADER + align256(rows * 4) + align256(rows * nb * f * 8);
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
    size_t off = WS_HEADER;
    P.counter = reinterpret_cast<unsigned *>(ws + off);
    off += align256(static_cast<size_t>(L.B) * L.K1 * 4);
    P.cand = reinterpret_cast<uint64_t *>(ws + off);
    P.draft = static_cast<const unsigned char *>(L.draft);
    P.exclude = L.exclude;
    P.out_ids = L.out_ids;
    P.row_status = L.row_status;
    return L.dtype == 0 ? launch_fan<FanoutOp<0>, 0>(P, L.tma, st) : launch_fan<FanoutOp<1>, 1>(P, L.tma, st);
}

}  // namespace spv
