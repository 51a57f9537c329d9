// spv_stream.cuh -- device building blocks of libspv (sm_103a).
//
// * A streaming pipeline that reads every logit row of a call exactly once:
//   rows are cut into work items of 8192 contiguous logits; a producer warp
//   stages items in a ring of shared-memory buffers with TMA bulk copies
//   (cp.async.bulk, global -> shared, completion on an mbarrier), and eight
//   consumer warps reduce one sampler block (1024 logits) each.  After a
//   few static items per CTA, the items are handed out by a per-call counter
//   in the workspace header, so faster CTAs take more of them.  Per-block
//   partial results go to a small workspace.  A second, dependent grid (one
//   CTA per sequence or row, or a cluster of them; programmatic dependent
//   launch) merges them and writes the outputs, so no streaming CTA ever
//   waits on another's work.  Optional per-op hooks: rows skipped by
//   producer and consumers alike, a per-call reset.
// * Philox4x32-10 and the uniform / exponential variates of the sampling rule.
// * Warp reductions, order-preserving float keys, packed fp32-pair arithmetic.
// * Bounded waits: on an mbarrier, on a flag, and a barrier of the CTAs of one
//   thread-block cluster through global memory.
//
// Every wait is bounded; a wait that gives up records SPV_ERR_TIMEOUT in the
// workspace error word and the CTA stops cleanly.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

namespace spv {

constexpr int G = 1024;                       // sampler block: tokens per block
constexpr int CHUNK_BLOCKS = 8;               // sampler blocks per work item
constexpr int CHUNK = G * CHUNK_BLOCKS;       // logits per work item
constexpr int NCW = 8;                        // consumer warps (one block each)
constexpr int THREADS = (NCW + 1) * 32;       // + one producer warp
constexpr int RING_BYTES_PER_SM = 192 * 1024; // shared-memory ring of all resident CTAs of an SM
constexpr uint32_t WAIT_LIMIT = 1u << 22;     // try_wait polls before giving up
constexpr int SKIP_TABLE_MAX = 1024;          // sequences whose row-skip table fits shared memory (8 KB)
constexpr int MAX_TRIALS = 64;                // residual rejection trials
constexpr int STATUS_BAD_ROW = 4;
constexpr int STATUS_TIMEOUT = 5;

constexpr int SUB = 32;                       // sampler sub-block: ids per sub-block

// Philox stream tags (second counter word).
constexpr uint32_t STREAM_BLOCK = 1, STREAM_SUB = 2, STREAM_TOKEN = 3, STREAM_ACCEPT = 4, STREAM_FB_BLOCK = 5,
                   STREAM_FB_SUB = 6, STREAM_FB_TOKEN = 7;

// Speculation-cache lookup fused into the verify finalize ([SSD] Algorithm 1,
// "if verify_outcome in cache"; Figure 2).  The cache of sequence b is its
// fan-out candidate list: for each position k = 0..gamma, F_k candidate
// tokens, k-major (the layout spv_fanout_topk writes).  The verify outcome
// (k accepted, emitted token t) hits the entry of position k that holds t.
constexpr int CACHE_POSITIONS = 33;  // gamma + 1 positions at most
struct CacheLookup {
    const int32_t *ids;              // [B, n] candidate ids, or null: no lookup
    int32_t *slot;                   // [B] out: entry index in the row of ids, -1 = miss or bad row
    int n;                           // sum_k F_k
    int off[CACHE_POSITIONS + 1];    // off[k] = sum_{j<k} F_j
};

// Pull sequence b's candidate row towards L2 (inputs: safe before the
// dependent-grid wait).  One warp.
__device__ __forceinline__ void cache_prefetch(const CacheLookup &C, int b, int lane)
{
    if (!C.ids) return;
    const char *base = reinterpret_cast<const char *>(C.ids + static_cast<size_t>(b) * C.n);
    for (int o = lane * 128; o < C.n * 4; o += 32 * 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(base + o));
}

// Slot of the outcome (k, t) of sequence b (k < 0: bad row, no hit).  One
// warp; candidate lists hold distinct ids, the lowest matching entry wins
// otherwise.
__device__ __forceinline__ void cache_lookup(const CacheLookup &C, int b, int k, int t, int lane)
{
    if (!C.ids) return;
    int slot = -1;
    if (k >= 0) {
        const int o0 = C.off[k], n = C.off[k + 1] - o0;
        const int32_t *row = C.ids + static_cast<size_t>(b) * C.n + o0;
        for (int j0 = 0; j0 < n; j0 += 32) {
            const int j = j0 + lane;
            const unsigned m = __ballot_sync(0xffffffffu, j < n && __ldg(row + j) == t);
            if (m) {
                slot = o0 + j0 + __ffs(m) - 1;
                break;
            }
        }
    }
    if (lane == 0) C.slot[b] = slot;
}

template <int DT> struct DType;
template <> struct DType<0> {  // fp32
    using T = float;
    static constexpr int BYTES = 4;
    __device__ static __forceinline__ float load(const void *p, long long i) {
        return __ldg(reinterpret_cast<const float *>(p) + i);
    }
};
template <> struct DType<1> {  // bf16
    using T = __nv_bfloat16;
    static constexpr int BYTES = 2;
    __device__ static __forceinline__ float load(const void *p, long long i) {
        unsigned short b = __ldg(reinterpret_cast<const unsigned short *>(p) + i);
        return __uint_as_float(static_cast<uint32_t>(b) << 16);
    }
};

// Ring stages of one CTA when `ctas` CTAs share an SM (at least 2), for work
// items of `chunk` logits.
template <int DT> constexpr int stages(int ctas, int chunk = CHUNK)
{
    return RING_BYTES_PER_SM / ctas / (chunk * DType<DT>::BYTES) < 2
               ? 2
               : RING_BYTES_PER_SM / ctas / (chunk * DType<DT>::BYTES);
}

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase of `parity` to complete; false if it gave up.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity)
{
    for (uint32_t i = 0; i < WAIT_LIMIT; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Whether a bounded wait gave up on this workspace: the error word holds
// STATUS_TIMEOUT (set by this call's streaming grid, or by an earlier call on
// the same workspace until it is zero-filled).  Read after the dependent-grid
// wait, so the streaming grid's writes are visible.
__device__ __forceinline__ bool workspace_timed_out(const unsigned *err)
{
    return *reinterpret_cast<const volatile unsigned *>(err) == static_cast<unsigned>(STATUS_TIMEOUT);
}

// Bounded wait until *flag >= target (acquire loads, short sleeps between
// polls); false, with STATUS_TIMEOUT in *err, after `limit` polls.
__device__ __forceinline__ bool wait_flag_ge(const unsigned *flag, unsigned target, uint32_t limit, unsigned *err)
{
    for (uint32_t i = 0; ld_acquire_gpu(flag) < target; ++i) {
        if (i == limit) {
            atomicExch(err, STATUS_TIMEOUT);
            return false;
        }
        __nanosleep(32);
    }
    return true;
}

// Barrier of the n CTAs of one thread-block cluster (co-scheduled, so every
// one of them arrives) through global memory: *ctr counts the arrivals of
// all the group's barriers of the call (zeroed before the group starts), so
// the group's j-th barrier (from 0) is complete once it reaches n (j + 1).
// One atomic per CTA and acquire polls by the waiting ones, no reset.  Called
// by all `threads` threads of each CTA (named barrier 1); global writes that
// each writer fenced (__threadfence) before it are visible to every CTA after
// it.  The wait is bounded: false (and STATUS_TIMEOUT in *err) if it gave up.
template <int THREADS_> __device__ __forceinline__ bool group_barrier(unsigned *ctr, unsigned n, unsigned j,
                                                                      unsigned *err, int *sh_flag)
{
    asm volatile("bar.sync 1, %0;" ::"n"(THREADS_) : "memory");
    if (threadIdx.x == 0) {
        const unsigned target = n * (j + 1u);
        __threadfence();
        int ok = 1;
        if (atomicAdd(ctr, 1u) + 1u < target) ok = wait_flag_ge(ctr, target, WAIT_LIMIT, err) ? 1 : 0;
        __threadfence();
        *sh_flag = ok;
    }
    asm volatile("bar.sync 1, %0;" ::"n"(THREADS_) : "memory");
    return *reinterpret_cast<volatile int *>(sh_flag) != 0;
}

// 16-byte asynchronous copy global -> shared by the executing thread (both
// addresses 16-byte aligned), and its commit / wait groups.
__device__ __forceinline__ void cp_async16(void *dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// TMA bulk copy global -> shared of `bytes` (multiple of 16, both addresses
// 16-byte aligned), completing on `bar` with `bytes` transaction count.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                         uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void consumer_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(NCW * 32) : "memory");
}

// Packed fp32 pairs (.f32x2 arithmetic, one instruction for two lanes of
// work): pack / unpack a pair and its FMA / add, each element rounded as the
// scalar operation would be.
__device__ __forceinline__ unsigned long long pack2(float lo, float hi)
{
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unpack2(unsigned long long v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long ffma2(unsigned long long a, unsigned long long b, unsigned long long c)
{
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ unsigned long long mul2(unsigned long long a, unsigned long long b)
{
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long fadd2(unsigned long long a, unsigned long long b)
{
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// max that propagates NaN (PTX max.NaN): one instruction per logit both
// finds the largest logit and flags NaN.
__device__ __forceinline__ float max_nan(float a, float b)
{
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ------------------------------------------------------------------ warp reductions
__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Warp max in one instruction (redux.sync, sm_100 and later): NaN inputs are
// ignored like fmaxf; every lane gets the result.
__device__ __forceinline__ float warp_max_redux(float v)
{
    float r;
    asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

// Max of three in one instruction (sm_100 and later); NaN ignored like fmaxf.
__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// argmax of (score, index): larger score wins, ties go to the lower index.
__device__ __forceinline__ void warp_argmax(float &s, int &i)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        int i2 = __shfl_xor_sync(0xffffffffu, i, o);
        if (s2 > s || (s2 == s && i2 < i)) {
            s = s2;
            i = i2;
        }
    }
}

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        uint64_t w = __shfl_xor_sync(0xffffffffu, v, o);
        v = w > v ? w : v;
    }
    return v;
}

// Order-preserving 32-bit key of a float (NaN excluded by the caller);
// -0.0 maps like +0.0.  Every key of a non-NaN float is >= 0x007FFFFF.
__device__ __forceinline__ uint32_t float_key(float x)
{
    uint32_t b = __float_as_uint(x);
    if (b == 0x80000000u) b = 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// ------------------------------------------------------------------ Philox4x32-10
// Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3"
// (SC'11): ten rounds; each multiplies counter words 0 and 2 by two 32-bit
// constants and mixes the 64-bit products' halves with the other words and
// the key, which is bumped by two Weyl constants between rounds.
__device__ __forceinline__ void philox4x32_10(uint32_t c[4], uint32_t k0, uint32_t k1)
{
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        if (round) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint32_t lo0 = 0xD2511F53u * c[0], hi0 = __umulhi(0xD2511F53u, c[0]);
        const uint32_t lo1 = 0xCD9E8D57u * c[2], hi1 = __umulhi(0xCD9E8D57u, c[2]);
        const uint32_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
        c[0] = n0;
        c[1] = lo1;
        c[2] = n2;
        c[3] = lo0;
    }
}

// The four words of draw group `grp` (draws 4*grp .. 4*grp+3) of one
// stream: counter (grp, stream, trial, 0), key (low, high half of `key`).
// The position a draw is made at is not part of the counter: a sequence
// makes one draw, so its variates can be generated before the position (the
// first rejection) is known.
__device__ __forceinline__ void philox_group(uint32_t w[4], uint64_t key, uint32_t stream, uint32_t trial,
                                             uint32_t grp)
{
    w[0] = grp;
    w[1] = stream;
    w[2] = trial;
    w[3] = 0u;
    philox4x32_10(w, static_cast<uint32_t>(key), static_cast<uint32_t>(key >> 32));
}

// U = ((w >> 8) + 1) * 2^-24 in (0, 1], exact in fp32.
__device__ __forceinline__ float uniform24(uint32_t w)
{
    return static_cast<float>((w >> 8) + 1u) * 0x1p-24f;
}

// E = -ln U in [0, 16.64] (0 when U == 1: an arrival at time zero).
__device__ __forceinline__ float expo(uint32_t w)
{
    return -logf(uniform24(w));
}

// Arrival time E * f of a candidate whose mass is 1/f (f may be +inf for a
// vanishing mass); E == 0 arrives at 0.
__device__ __forceinline__ float arrival(float E, float f)
{
    return E == 0.f ? 0.f : E * f;
}

// argmin of (arrival, index) across the warp, ties to the lower index, for
// arrivals >= 0 or +inf (never NaN): their bit patterns order like their
// values, so two single-instruction reductions replace a shuffle tree (the
// draws run on one warp, where every step of a dependent chain counts).
__device__ __forceinline__ void warp_argmin(float &a, int &i)
{
    const unsigned ab = __float_as_uint(a) & 0x7fffffffu;  // -0.0 ranks as +0.0
    const unsigned mn = __reduce_min_sync(0xffffffffu, ab);
    i = static_cast<int>(__reduce_min_sync(0xffffffffu, ab == mn ? static_cast<unsigned>(i) : 0xffffffffu));
    a = __uint_as_float(mn);
}

// ------------------------------------------------------------------ block loads
// Lane `lane` owns 32 logits of a 1024-logit block; element e of the lane is
// block index idx(e).  fp32: 8 x float4 at j*128 + lane*4; bf16: 4 x 8 at
// j*256 + lane*8.  Both orders rise with e.
template <int DT> __device__ __forceinline__ int lane_index(int lane, int e)
{
    if (DT == 0) return (e >> 2) * 128 + lane * 4 + (e & 3);
    return (e >> 3) * 256 + lane * 8 + (e & 7);
}

// From shared memory (16-byte vector loads; the block starts 16-byte aligned).
template <int DT> __device__ __forceinline__ void load_block_smem(float v[32], const unsigned char *blk, int lane)
{
    if (DT == 0) {
        const float4 *p = reinterpret_cast<const float4 *>(blk);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float4 t = p[j * 32 + lane];
            v[4 * j] = t.x;
            v[4 * j + 1] = t.y;
            v[4 * j + 2] = t.z;
            v[4 * j + 3] = t.w;
        }
    } else {
        const uint4 *p = reinterpret_cast<const uint4 *>(blk);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint4 t = p[j * 32 + lane];
            const uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                v[8 * j + 2 * h] = __uint_as_float(w[h] << 16);
                v[8 * j + 2 * h + 1] = __uint_as_float(w[h] & 0xffff0000u);
            }
        }
    }
}

// Elements of a partial block (index >= valid) become -inf.
template <int DT> __device__ __forceinline__ void mask_tail(float v[32], int valid, int lane)
{
    if (valid < G) {
#pragma unroll
        for (int e = 0; e < 32; ++e)
            if (lane_index<DT>(lane, e) >= valid) v[e] = -INFINITY;
    }
}

// From global memory, scalar loads (any alignment); elements >= valid are -inf.
template <int DT>
__device__ __forceinline__ void load_block_global(float v[32], const void *blk, int lane, int valid)
{
#pragma unroll
    for (int e = 0; e < 32; ++e) {
        const int i = lane_index<DT>(lane, e);
        v[e] = i < valid ? DType<DT>::load(blk, i) : -INFINITY;
    }
}

// ------------------------------------------------------------------ item positions
// Quotient of a row index by a small positive divisor: 32-bit unsigned
// division while the row fits in 32 bits (every call in practice), else the
// 64-bit one.
__device__ __forceinline__ long long div_row(long long row, int d)
{
    return row <= 0xffffffffLL ? static_cast<long long>(static_cast<uint32_t>(row) / static_cast<uint32_t>(d))
                               : row / d;
}

// The work-item counter of a call: 64 bits at byte 8 of the workspace header
// (after the error word and the self-test flag).  Zero between calls: a
// zero-filled workspace starts it at 0 and every finalize grid returns it to 0.
__device__ __forceinline__ unsigned long long *item_counter(unsigned *err)
{
    return reinterpret_cast<unsigned long long *>(err + 2);
}

// Position (row, chunk c) of work item it = row * nc + c, advanced by a fixed
// stride of items without a division per step.
struct ItemPos {
    long long row;
    int c;
    int nc, dq, dr;  // items per row; stride = dq * nc + dr
    __device__ __forceinline__ ItemPos(unsigned first, unsigned stride, int nc_)
        : row(first / static_cast<unsigned>(nc_)), c(static_cast<int>(first % static_cast<unsigned>(nc_))), nc(nc_),
          dq(static_cast<int>(stride / static_cast<unsigned>(nc_))),
          dr(static_cast<int>(stride % static_cast<unsigned>(nc_))) {}
    // Row of the item one stride ahead.
    __device__ __forceinline__ long long next_row() const { return row + dq + (c + dr >= nc ? 1 : 0); }
    __device__ __forceinline__ void advance()
    {
        row += dq;
        c += dr;
        if (c >= nc) {
            c -= nc;
            ++row;
        }
    }
};

// ------------------------------------------------------------------ the pipeline
// Op supplies:
//   struct Params  -- with total_items, nc (items per row), nb (blocks per
//                     row), V and err fields;
//   CTAS_PER_SM                          resident CTAs the kernel is built for;
//   row_ptr(P, row)                      global address of a row;
//   block(P, row, beta, v, valid, lane)  per-warp reduction of one block
//                                        (32 logits per lane as floats);
//   block_smem(P, row, beta, blk, valid, lane)  the same from the staged
//                                        block in shared memory;
//   finalize(P, g, sm, warp, lane)       merge + outputs of group g (run by
//                                        finalize_kernel, one CTA per group);
//   struct Smem                          shared scratch of finalize.
// and optionally (SKIPS = true) rows it does not read at all:
//   skip_key(P, row, lane)               a per-lane input of skip(), read
//                                        from global memory one item ahead;
//   skip(P, row, key, lane)              warp-uniform: the row is skipped;
//   reset(P)                             run by every thread at the start;
//   TABLE                                number the items over the rows read
//                                        instead (rows staged by TMA, at most
//                                        SKIP_TABLE_MAX sequences), with
//   build_table(P, mask, first)          the CTA's table of rows read, and
//   item_row(P, mask, first, it, nc, row, c)  the row and chunk of item it.
// Producer and consumers take the same decisions, so a skipped item uses
// no ring stage; with the table the skipped rows have no items at all and
// the producer hands items out through the call's counter.
// and optionally (WAITS_PRIOR = true) the consumers wait for the grid
// launched before this one (programmatic dependent launch): the producer's
// copies start while that grid finishes.
template <class Op, class = void> struct OpWaitsPrior {
    static constexpr bool value = false;
};
template <class Op> struct OpWaitsPrior<Op, std::void_t<decltype(Op::WAITS_PRIOR)>> {
    static constexpr bool value = Op::WAITS_PRIOR;
};

// Sampler blocks per work item (Op::ITEM_BLOCKS, a multiple of the consumer
// warps, else CHUNK_BLOCKS): each consumer warp reduces ITEM_BLOCKS / NCW
// blocks of a staged item.
template <class Op, class = void> struct OpItemBlocks {
    static constexpr int value = CHUNK_BLOCKS;
};
template <class Op> struct OpItemBlocks<Op, std::void_t<decltype(Op::ITEM_BLOCKS)>> {
    static constexpr int value = Op::ITEM_BLOCKS;
};

template <class Op, class = void> struct OpSkips {
    static constexpr bool value = false;
};
template <class Op> struct OpSkips<Op, std::void_t<decltype(Op::SKIPS)>> {
    static constexpr bool value = Op::SKIPS;
};

template <class Op, int DT, bool TMA>
__global__ void __launch_bounds__(THREADS, Op::CTAS_PER_SM) stream_kernel(const typename Op::Params P)
{
    constexpr int EB = DType<DT>::BYTES;
    constexpr int CB = OpItemBlocks<Op>::value;  // blocks per work item
    static_assert(CB % NCW == 0, "work items hold a whole number of blocks per consumer warp");
    constexpr int CH = G * CB;                   // logits per work item
    constexpr int S = stages<DT>(Op::CTAS_PER_SM, CH);
    constexpr int CHUNK_BYTES = CH * EB;
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ __align__(8) uint64_t full_bar[S];
    __shared__ __align__(8) uint64_t empty_bar[S];
    __shared__ long long stage_row[S];  // item of each ring stage (dynamic assignment): row, -1 = no more
    __shared__ int stage_c[S];          // and chunk
    __shared__ volatile int sh_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], NCW);
        }
        sh_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // The dependent finalize grid may be scheduled as soon as resources free
    // up; it waits (griddepcontrol.wait) for this grid's results itself.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    long long total = P.total_items;
    const int nc = P.nc;
    constexpr bool SK = OpSkips<Op>::value;
    // A row-skipping op with staged rows, Op::TABLE and at most SKIP_TABLE_MAX sequences: the whole CTA
    // first builds a table of the rows it reads (per sequence: a bit per node, and the rows read
    // before the sequence), and the items are numbered over those rows alone; the producer then
    // hands them out through the call's counter like the other ops.  Otherwise every item of
    // every row is taken on the static stride with a warp vote on its row (skip_key / skip).
    __shared__ unsigned long long skip_mask[SK ? SKIP_TABLE_MAX : 1];
    __shared__ int skip_first[SK ? SKIP_TABLE_MAX + 1 : 1];
    bool table = false;
    if constexpr (SK) {
        Op::reset(P);
        table = TMA && Op::TABLE && P.B <= SKIP_TABLE_MAX;
        if (table) {
            Op::build_table(P, skip_mask, skip_first);  // ends with __syncthreads
            total = static_cast<long long>(skip_first[P.B]) * nc;
        }
    }

    if (warp == NCW) {  // ---------------- producer
        if constexpr (SK) {
            if (TMA && !table) {  // the whole warp walks the items (skip() is a warp vote); lane 0 copies
                const uint64_t pol = l2_evict_first_policy();
                int i = 0;
                long long it = blockIdx.x;
                ItemPos pos(blockIdx.x, gridDim.x, nc);
                int key = it < total ? Op::skip_key(P, pos.row, lane) : 0;
                for (; it < total; it += gridDim.x, pos.advance()) {
                    const long long row = pos.row;
                    const long long nx = it + gridDim.x;
                    const int nkey = nx < total ? Op::skip_key(P, pos.next_row(), lane) : 0;
                    const bool skip = Op::skip(P, row, key, lane);
                    key = nkey;
                    if (skip) continue;
                    const int s = i % S;
                    const uint32_t ph = (i / S) & 1;
                    int stop = 0;
                    if (lane == 0) {
                        if (!mbar_wait(&empty_bar[s], ph ^ 1u)) {
                            atomicExch(P.err, STATUS_TIMEOUT);
                            sh_abort = 1;
                            stop = 1;
                        } else if (sh_abort) {
                            stop = 1;
                        } else {
                            const int c = pos.c;
                            const int n = min(CH, P.V - c * CH);
                            const unsigned char *src = reinterpret_cast<const unsigned char *>(Op::row_ptr(P, row)) +
                                                       static_cast<size_t>(c) * CHUNK_BYTES;
                            mbar_arrive_expect_tx(&full_bar[s], static_cast<uint32_t>(n * EB));
                            bulk_g2s(ring + s * CHUNK_BYTES, src, static_cast<uint32_t>(n * EB), &full_bar[s], pol);
                        }
                    }
                    if (__shfl_sync(0xffffffffu, stop, 0)) break;
                    ++i;
                }
                if (lane == 0)
                    for (int k = max(0, i - S); k < i; ++k) mbar_wait(&full_bar[k % S], (k / S) & 1);
            }
            if (!table) return;
        }
        if (TMA && lane == 0) {
            // Work items: this CTA's first S are static (it = blockIdx.x + j * grid, j < S); the rest
            // are handed out in increasing order by the call's item counter, so the CTAs that stream
            // faster take more of them (with equal shares the slowest SMs set the end of the pass).
            // The next item's index is fetched one item ahead: the atomic's latency hides behind the
            // wait for a free stage.  Each stage carries its item's (row, chunk) to the consumers; the
            // stage after the last item carries row -1 and no copy.  (A row-skipping op numbers its
            // items over the rows it reads: table above.)
            const uint64_t pol = l2_evict_first_policy();
            unsigned long long *ctr = item_counter(P.err);
            const long long first_dyn = static_cast<long long>(S) * gridDim.x;
            // With fewer than 4 items per CTA left after the static ones, the counter's atomics (all
            // CTAs at once) cost more than the balance gains: keep the static stride for every item.
            const bool dyn = total - first_dyn >= 4LL * gridDim.x;
            int i = 0;
            bool aborted = false;
            for (long long it = blockIdx.x; it < total;) {
                const long long nx = (i + 1 < S || !dyn) ? blockIdx.x + static_cast<long long>(i + 1) * gridDim.x
                                                         : first_dyn + static_cast<long long>(atomicAdd(ctr, 1ull));
                const int s = i % S;
                const uint32_t ph = (i / S) & 1;
                if (!mbar_wait(&empty_bar[s], ph ^ 1u)) {
                    atomicExch(P.err, STATUS_TIMEOUT);
                    sh_abort = 1;
                    aborted = true;
                    break;
                }
                if (sh_abort) {
                    aborted = true;
                    break;
                }
                long long row;
                int c;
                if constexpr (SK) {
                    Op::item_row(P, skip_mask, skip_first, it, nc, row, c);
                } else {
                    row = div_row(it, nc);
                    c = static_cast<int>(it - row * nc);
                }
                stage_row[s] = row;
                stage_c[s] = c;
                const int n = min(CH, P.V - c * CH);
                const unsigned char *src =
                    reinterpret_cast<const unsigned char *>(Op::row_ptr(P, row)) + static_cast<size_t>(c) * CHUNK_BYTES;
                mbar_arrive_expect_tx(&full_bar[s], static_cast<uint32_t>(n * EB));
                bulk_g2s(ring + s * CHUNK_BYTES, src, static_cast<uint32_t>(n * EB), &full_bar[s], pol);
                ++i;
                it = nx;
            }
            // No copy may still be writing this CTA's shared memory at exit.  (Drained before the end
            // mark: the end mark completes one more phase of the stage of item i - S, after which a
            // wait on that item's phase parity would name the next, never completed, phase.)
            for (int k = max(0, i - S); k < i; ++k) mbar_wait(&full_bar[k % S], (k / S) & 1);
            if (!aborted) {
                const int s = i % S;
                if (mbar_wait(&empty_bar[s], ((i / S) & 1) ^ 1u)) {
                    stage_row[s] = -1;
                    mbar_arrive(&full_bar[s]);
                } else {
                    atomicExch(P.err, STATUS_TIMEOUT);
                    sh_abort = 1;
                }
            }
        }
        return;
    }

    // ---------------- consumers
    if constexpr (OpWaitsPrior<Op>::value) asm volatile("griddepcontrol.wait;" ::: "memory");
    if (TMA && (!SK || table)) {  // the items the producer hands over, stage by stage
        int stage = 0;
        uint32_t phase = 0;
        for (;;) {
            if (!mbar_wait(&full_bar[stage], phase)) {
                atomicExch(P.err, STATUS_TIMEOUT);
                sh_abort = 1;
                break;
            }
            const long long row = stage_row[stage];
            if (row < 0) break;  // no more items (the end mark holds no copy to release)
#pragma unroll
            for (int q = warp; q < CB; q += NCW) {
                const int beta = stage_c[stage] * CB + q;
                if (beta < P.nb)
                    Op::block_smem(P, row, beta, ring + stage * CHUNK_BYTES + q * G * EB, min(G, P.V - beta * G),
                                   lane);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[stage]);
            // A timed-out wait anywhere stops every consumer warp together.
            if (__any_sync(0xffffffffu, sh_abort != 0)) break;
            if (++stage == S) {
                stage = 0;
                phase ^= 1u;
            }
        }
        return;
    }
    int i = 0;
    int key = 0;
    ItemPos pos(blockIdx.x, gridDim.x, nc);
    if constexpr (SK) key = blockIdx.x < total ? Op::skip_key(P, pos.row, lane) : 0;
    for (long long it = blockIdx.x; it < total; it += gridDim.x, pos.advance()) {
        if constexpr (SK) {
            const long long nx = it + gridDim.x;
            const int nkey = nx < total ? Op::skip_key(P, pos.next_row(), lane) : 0;
            const bool skip = Op::skip(P, pos.row, key, lane);
            key = nkey;
            if (skip) continue;
        }
        const int s = i % S;
        const uint32_t ph = (i / S) & 1;
        bool ok = true;
        if (TMA) {
            ok = mbar_wait(&full_bar[s], ph);
            if (!ok) {
                atomicExch(P.err, STATUS_TIMEOUT);
                sh_abort = 1;
            }
        }
        const long long row = pos.row;
        const int c = pos.c;
#pragma unroll
        for (int q = warp; q < CB; q += NCW) {
            const int beta = c * CB + q;
            if (ok && beta < P.nb) {
                const int valid = min(G, P.V - beta * G);
                if (TMA) {
                    Op::block_smem(P, row, beta, ring + s * CHUNK_BYTES + q * G * EB, valid, lane);
                } else {
                    float v[32];
                    const unsigned char *blk = reinterpret_cast<const unsigned char *>(Op::row_ptr(P, row)) +
                                               static_cast<size_t>(beta) * G * EB;
                    load_block_global<DT>(v, blk, lane, valid);
                    Op::block(P, row, beta, v, valid, lane);
                }
            }
        }
        if (TMA) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[s]);
            // A timed-out wait anywhere stops every consumer warp together.
            if (__any_sync(0xffffffffu, sh_abort != 0)) break;
        }
        ++i;
    }
}

// One CTA (Op::FIN_WARPS warps) per group: merges the group's partial results once the
// streaming grid it depends on has finished, and writes the outputs.
template <class Op, int DT>
__global__ void __launch_bounds__(Op::FIN_WARPS * 32, 1) __maxnreg__(Op::FIN_WARPS >= 32 ? 64 : (Op::FIN_WARPS >= 16 ? 96 : 128)) finalize_kernel(const typename Op::Params P)
{
    __shared__ typename Op::Smem sm;
    extern __shared__ __align__(16) float fin_buf[];  // Op::FIN_BUF_FLOATS floats
    // Op::finalize issues griddepcontrol.wait before it reads anything the
    // streaming grid wrote; reads of the call's inputs may come before it.
    Op::finalize(P, static_cast<int>(blockIdx.x), sm, fin_buf, threadIdx.x >> 5, threadIdx.x & 31);
    // The streaming grid has completed once the dependent-grid wait returns:
    // return the call's work-item counter to zero for the next call.
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        *item_counter(P.err) = 0ull;
    }
}

// SM count of the current device (queried once per device).
static inline cudaError_t device_sm_count(int *out)
{
    constexpr int MAX_DEV = 64;
    static int cache[MAX_DEV];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < MAX_DEV && cache[dev] > 0) {
        *out = cache[dev];
        return cudaSuccess;
    }
    int sms = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if (dev >= 0 && dev < MAX_DEV) cache[dev] = sms;
    *out = sms;
    return cudaSuccess;
}

// Launches the streaming grid of Op (persistent: as many CTAs as fit, capped
// by the item count) and then the finalize grid of Fin, `groups` CTAs, as a
// programmatic dependent launch on the same stream.
template <class Op, class Fin, int DT>
static cudaError_t launch_stream_finalize(const typename Op::Params &P0, bool tma, int groups, cudaStream_t st,
                                          int cluster = 1)
{
    constexpr bool PRIOR = OpWaitsPrior<Op>::value;
    constexpr int CH = G * OpItemBlocks<Op>::value;
    // Work items of this op: P0 counts them in items of CHUNK logits.
    typename Op::Params P = P0;
    const long long rows = P0.total_items / P0.nc;
    P.nc = (P0.V + CH - 1) / CH;
    P.total_items = rows * P.nc;
    void (*kern)(const typename Op::Params) = tma ? stream_kernel<Op, DT, true> : stream_kernel<Op, DT, false>;
    const int smem = tma ? stages<DT>(Op::CTAS_PER_SM, CH) * CH * DType<DT>::BYTES : 0;
    // Per device and kernel variant: the shared-memory attributes and the
    // resident CTA count are set / queried once (the function-local static
    // is per template instantiation; the TMA / plain-load variant is chosen
    // at run time, so it indexes the cache).
    constexpr int MAX_DEV = 64;
    static int cap_cache[2][MAX_DEV];  // [TMA variant][device]: resident CTAs of the GPU, 0 = not yet known
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int *slot = (dev >= 0 && dev < MAX_DEV) ? &cap_cache[tma ? 1 : 0][dev] : nullptr;
    int cap = slot ? *slot : 0;
    if (cap == 0) {
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
            return e;
        int sms = 0, per_sm = 0;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, THREADS, smem)) != cudaSuccess)
            return e;
        cap = (per_sm < 1 ? 1 : per_sm) * sms;
        if ((e = cudaFuncSetAttribute(finalize_kernel<Fin, DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      Fin::FIN_BUF_FLOATS * 4)) != cudaSuccess)
            return e;
        if (slot) *slot = cap;
    }
    const int grid = static_cast<int>(P.total_items < cap ? P.total_items : cap);
    if (PRIOR) {  // a programmatic dependent launch on the grid before it
        cudaLaunchConfig_t sc = {};
        sc.gridDim = dim3(static_cast<unsigned>(grid));
        sc.blockDim = dim3(THREADS);
        sc.dynamicSmemBytes = static_cast<size_t>(smem);
        sc.stream = st;
        cudaLaunchAttribute sa[1];
        sa[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        sa[0].val.programmaticStreamSerializationAllowed = 1;
        sc.attrs = sa;
        sc.numAttrs = 1;
        if ((e = cudaLaunchKernelEx(&sc, kern, P)) != cudaSuccess) return e;
    } else {
        kern<<<grid, THREADS, smem, st>>>(P);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(groups));
    cfg.blockDim = dim3(Fin::FIN_WARPS * 32);
    cfg.dynamicSmemBytes = Fin::FIN_BUF_FLOATS * 4;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cluster > 1) {  // finalize CTAs g*cluster .. g*cluster+cluster-1 co-scheduled as one cluster
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = static_cast<unsigned>(cluster);
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, finalize_kernel<Fin, DT>, P);
}

}  // namespace spv
