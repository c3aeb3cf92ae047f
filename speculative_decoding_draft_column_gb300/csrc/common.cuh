// Device pieces shared by the two streaming kernels of libspecsel: the
// round's arguments, bf16 order keys and packed entries, bf16x2 max trees and
// compares, masked edge loads, mbarrier / bulk-copy primitives with bounded
// waits, candidate-buffer pruning and the flat-run slicing.
//
// The operations ("A drafter inside the artifact", Ignis DFlash2 page,
// section "How it works"): top-k over each draft column (largest first, ties
// to the smaller token id) and greedy verify (per target column the argmax,
// then per lane the longest matching draft prefix plus the bonus token).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "specsel.h"

namespace {

constexpr uint64_t kWaitLimitNs = 4000000000ull;   // bound on any mbarrier wait: 4 s of wall time
constexpr unsigned kFull = 0xffffffffu;
constexpr uint32_t kNaN2 = 0x7FFF7FFFu;            // two bf16 NaNs: the mask value

struct RoundArgs {
    // top-k part (draft columns)
    const uint16_t *draft;
    int64_t d_cols, d_V;
    int32_t k;
    const int32_t *id_map;
    uint16_t *out_vals;
    int32_t *out_ids;
    // verify part (target columns)
    const uint16_t *target;
    int64_t t_cols, t_V;
    int32_t gamma;
    const int32_t *drafts;
    int32_t *out_accept;
    int32_t *out_commit;
    // streaming units (warps or CTAs, by kernel): [0, d_units) stream the
    // draft logits, [d_units, d_units + t_units) the target logits
    int32_t d_units, t_units;
    // scratch
    unsigned long long *partials;   // [(d_units + t_units) * 2][pstride]: published lists
    unsigned int *col_ticket;       // [d_cols + t_cols]
    unsigned int *col_cert;         // [d_cols + t_cols]: best certified key published for a split column
    unsigned int *lane_ticket;      // [lanes]: the lane's finished columns (per-warp kernel); with, from
                                    // bit 8 on, a bit per matching draft (CTA kernel)
    int32_t pstride;
    uint16_t *gkeys;                // group-maxima kernel: group keys of both runs (in the partials area)
    spec_counters *counters;        // null: no counting
    // sampled verify (uniforms non-null): the target columns keep their
    // top t_k (else t_k = 1, the argmax)
    int32_t t_k;
    double temperature, top_p;
    const double *uniforms;         // [lanes][gamma+1][2]
};

__device__ __forceinline__ uint32_t atom_add_acq_rel(unsigned int *p, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Add one verified lane's outcome (accept length acc of gamma drafts) to the
// round counters: one lane per position (device atomics).
__device__ __forceinline__ void count_lane(spec_counters *cnt, int gamma, int acc, int lane)
{
    if (!cnt) return;
    if (lane == 0) {
        atomicAdd(reinterpret_cast<unsigned long long *>(&cnt->rounds), 1ull);
        atomicAdd(reinterpret_cast<unsigned long long *>(&cnt->drafted_tokens), (unsigned long long)gamma);
        atomicAdd(reinterpret_cast<unsigned long long *>(&cnt->accepted_tokens), (unsigned long long)acc);
    }
    if (lane < gamma) {
        atomicAdd(reinterpret_cast<unsigned long long *>(&cnt->position_drafted[lane]), 1ull);
        if (lane < acc) atomicAdd(reinterpret_cast<unsigned long long *>(&cnt->position_accepted[lane]), 1ull);
    }
}

// Set (bit 0) when a bounded wait gave up; read and cleared by spec_device_status.
__device__ unsigned int g_wait_timeouts;

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// true if either bf16 half of a is > (or >=) the bf16 in both halves of t2;
// NaN halves compare false.
__device__ __forceinline__ bool any_gt(uint32_t a, uint32_t t2)
{
    uint32_t r;
    asm("{\n\t.reg .pred p, q;\n\t"
        "setp.gt.bf16x2 p|q, %1, %2;\n\t"
        "or.pred p, p, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(a), "r"(t2));
    return r != 0;
}

__device__ __forceinline__ bool any_ge(uint32_t a, uint32_t t2)
{
    uint32_t r;
    asm("{\n\t.reg .pred p, q;\n\t"
        "setp.ge.bf16x2 p|q, %1, %2;\n\t"
        "or.pred p, p, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(a), "r"(t2));
    return r != 0;
}

// a / b for a >= 0, b > 0: the 32-bit divide when both fit in 32 bits (a
// handful of instructions), the 64-bit routine (several times longer) only
// otherwise.  The indices divided here (columns, lanes, CTAs, vectors of
// rounds below 2^32 of them) nearly always fit.
__device__ __forceinline__ int64_t udiv(int64_t a, int64_t b)
{
    if ((((uint64_t)a | (uint64_t)b) >> 32) == 0) return (int64_t)((uint32_t)a / (uint32_t)b);
    return a / b;
}

__device__ __forceinline__ float bf16_as_float(uint32_t raw16) { return __uint_as_float(raw16 << 16); }

// element e (0..7) of a 16-byte vector, widened exactly to float
__device__ __forceinline__ float elem8(const uint4 &q, int e)
{
    const uint32_t w = (e & 4) ? ((e & 2) ? q.w : q.z) : ((e & 2) ? q.y : q.x);
    return __uint_as_float((e & 1) ? (w & 0xFFFF0000u) : (w << 16));
}

// order-preserving 16-bit key of a bf16: -0 and +0 share a key; -Inf -> 0x80;
// NaN (the mask value) -> 0, below every real key.
__device__ __forceinline__ uint32_t order_key(uint32_t raw16)
{
    const uint32_t m = raw16 & 0x7FFFu;
    if (m > 0x7F80u) return 0u;
    return (raw16 & 0x8000u) ? (0x8000u - m) : (0x8000u + m);
}

__device__ __forceinline__ uint32_t key_to_raw(uint32_t key)
{
    const int s = (int)key - 0x8000;
    return s >= 0 ? (uint32_t)s : (0x8000u | (uint32_t)(-s));
}

// larger packed value = better entry: (key desc, id asc); low 16 bits keep the
// element's own bit pattern (so -0 survives); 0 = empty slot.
__device__ __forceinline__ unsigned long long pack_entry(float v, uint32_t id)
{
    if (v != v) return 0ull;
    const uint32_t raw = __float_as_uint(v) >> 16;
    return ((unsigned long long)order_key(raw) << 48) | ((unsigned long long)(~id) << 16) | raw;
}

__device__ __forceinline__ uint32_t entry_key(unsigned long long e) { return (uint32_t)(e >> 48); }
__device__ __forceinline__ uint32_t entry_id(unsigned long long e) { return ~(uint32_t)(e >> 16); }
__device__ __forceinline__ uint16_t entry_raw(unsigned long long e) { return (uint16_t)(e & 0xFFFFu); }

// bf16x2 max over one 16-byte vector
__device__ __forceinline__ uint32_t vmax(const uint4 &q) { return bmax2(bmax2(q.x, q.y), bmax2(q.z, q.w)); }

// both halves hold max(lo, hi)
__device__ __forceinline__ uint32_t hmax_splat(uint32_t m2) { return bmax2(m2, __byte_perm(m2, 0, 0x1032)); }

// Masked load of an edge vector: element by element, only inside [g0, g1).
__device__ __forceinline__ uint4 load_edge(const uint16_t *buf, int64_t j, int mis, int64_t g0, int64_t g1)
{
    uint32_t w[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        uint32_t lo = 0x7FFFu, hi = 0x7FFFu;
        const int64_t ga = 8 * j + 2 * h - mis, gb = ga + 1;
        if (ga >= g0 && ga < g1) lo = __ldg(buf + ga);
        if (gb >= g0 && gb < g1) hi = __ldg(buf + gb);
        w[h] = lo | (hi << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ uint32_t lanemask_lt()
{
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Exclusive prefix sum of v over the warp; also returns the warp total.
__device__ __forceinline__ int warp_exclusive_sum(int v, int lane, int &total)
{
    int incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(kFull, incl, d);
        if (lane >= d) incl += y;
    }
    total = __shfl_sync(kFull, incl, 31);
    return incl - v;
}

// A 32-bit word other SMs update with atomics, read through L2.
__device__ __forceinline__ uint32_t ld_relaxed(const unsigned int *p)
{
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Programmatic dependent launch: let the next launch on the stream be
// scheduled now (its CTAs still wait below for this grid to finish), and
// wait for the previous launch to finish and flush before touching memory.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---- mbarrier / bulk-copy primitives (inline PTX, sm_90+) -------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// Test the phase; a thread whose phase is not complete may sleep in the
// instruction until it completes (at most the hinted 20 us), instead of
// spinning on the issue slots.
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(smem_u32(bar)), "r"(parity), "n"(20000)
                 : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Set by a thread of the CTA whose wait gave up: the CTA's other waits then
// give up at once, so a launch ends within one time limit.
__shared__ unsigned int s_gave_up;

// Wait for the phase with the given parity to complete, for at most
// limit_ns of wall time; on giving up, flag the error and report false (the
// data is then garbage, but the kernel still terminates).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*reinterpret_cast<volatile unsigned int *>(&s_gave_up)) return false;
        if (global_ns() - t0 > limit_ns) {
            s_gave_up = 1u;
            atomicOr(&g_wait_timeouts, 1u);
            return false;
        }
    }
}


// One bulk copy global -> shared, completing on `bar` with its byte count.
// src, dst 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// ---- candidate buffers ------------------------------------------------------

struct Pruned {
    int n;       // entries kept (kk)
    uint32_t t;  // their certificate: the kk-th largest key
};

// Prune the buffer wb[0..n) (kk <= n <= 32 * Q, any order) to its kk best
// entries; returns kk and the kk-th largest key t (kk entries reach it: a
// certificate).  Ties at t go to the smallest ids (token ids, or mapped
// vocabulary ids for a shortlist), found by a bisection over the id bits only
// when there are more ties than places.
template <int Q>
__device__ __noinline__ Pruned buf_prune(unsigned long long *wb, int n, int kk, int lane)
{
    unsigned long long e[Q];
    uint32_t key[Q];
#pragma unroll
    for (int q = 0; q < Q; ++q) {
        const int idx = q * 32 + lane;
        e[q] = idx < n ? wb[idx] : 0ull;
        key[q] = entry_key(e[q]);
    }
    uint32_t t = 0;   // kk-th largest key: bisection over the 16 key bits
#pragma unroll 1
    for (int bit = 15; bit >= 0; --bit) {
        const uint32_t tr = t | (1u << bit);
        int cnt = 0;
#pragma unroll
        for (int q = 0; q < Q; ++q) cnt += __popc(__ballot_sync(kFull, key[q] >= tr));
        if (cnt >= kk) t = tr;
    }
    int cgt = 0, ceq = 0;
#pragma unroll
    for (int q = 0; q < Q; ++q) {
        cgt += __popc(__ballot_sync(kFull, key[q] > t));
        ceq += __popc(__ballot_sync(kFull, key[q] == t && e[q] != 0ull));
    }
    const int quota = kk - cgt;   // entries with key == t that survive
    uint32_t tid[Q];
#pragma unroll
    for (int q = 0; q < Q; ++q) tid[q] = (key[q] == t && e[q] != 0ull) ? entry_id(e[q]) : 0xFFFFFFFFu;
    uint32_t m = 0x7FFFFFFFu;     // ties kept: id <= m (ids < 2^31)
    if (ceq > quota) {
        m = 0;   // the quota-th smallest id among the ties
#pragma unroll 1
        for (int bit = 30; bit >= 0; --bit) {
            const uint32_t tr = m | (1u << bit);
            int cnt = 0;
#pragma unroll
            for (int q = 0; q < Q; ++q) cnt += __popc(__ballot_sync(kFull, tid[q] < tr));
            if (cnt < quota) m = tr;
        }
    }
    __syncwarp();
    int out = 0;
#pragma unroll
    for (int q = 0; q < Q; ++q) {
        const bool keep = key[q] > t || (tid[q] != 0xFFFFFFFFu && tid[q] <= m);
        const uint32_t bal = __ballot_sync(kFull, keep);
        if (keep) wb[out + __popc(bal & lanemask_lt())] = e[q];
        out += __popc(bal);
    }
    __syncwarp();
    return Pruned{out, t};
}

// Filter: candidates must be > thr (strict) or >= thr.
struct Filter {
    float thr;
    uint32_t thr2;   // thr as a bf16 pair
    bool strict;
};

// own_key: the warp's certified key for the column (0: none), strict unless
// mapped; cert_key: another certificate for the column (inclusive).
__device__ __forceinline__ Filter make_filter(uint32_t own_key, uint32_t cert_key, bool mapped)
{
    Filter f;
    uint32_t key;
    if (own_key != 0 && own_key >= cert_key) {
        key = own_key;
        f.strict = !mapped;
    } else {
        key = cert_key;
        f.strict = false;
    }
    const uint32_t raw = key ? key_to_raw(key) : 0xFF80u;   // no certificate: >= -Inf
    f.thr = bf16_as_float(raw);
    f.thr2 = raw | (raw << 16);
    return f;
}

__device__ __forceinline__ uint32_t elem_mask(const uint4 &q, const Filter &f)
{
    uint32_t cm = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const float v = elem8(q, e);
        cm |= (uint32_t)(f.strict ? (v > f.thr) : (v >= f.thr)) << e;
    }
    return cm;
}

// One buffer (draft or target logits) seen as a flat run of N = cols * V
// elements on the 16-byte vector grid: vector j holds elements
// [8j - mis, 8j - mis + 8).  The run is cut into W slices of whole vectors,
// one per streaming unit (a warp or a CTA); slice b = vectors
// [start(b), start(b+1)), start(b) = floor(b * NV / W).
struct Run {
    const uint16_t *buf;
    const uint4 *vb;          // 16-byte aligned base, at or just below buf
    int64_t V, N, NV;
    int64_t jlo, jhi;         // vectors [jlo, jhi) lie wholly inside the buffer
    int W, gw0;               // units on this run; global index of its slice 0
    int kk;
    int mis;
    bool draft;
};

__device__ __forceinline__ int64_t slice_start(const Run &r, int64_t w) { return udiv(w * r.NV, r.W); }
__device__ __forceinline__ int64_t owner(const Run &r, int64_t j) { return udiv((j + 1) * r.W - 1, r.NV); }
__device__ __forceinline__ int64_t first_elem(const Run &r, int64_t w)
{
    const int64_t g = 8 * slice_start(r, w) - r.mis;
    return g > 0 ? g : 0;
}

// The list slot of slice w for column c: 0 if c is the first column of the
// slice, else 1 (a slice holds part of at most two columns that it shares).
__device__ __forceinline__ unsigned long long *list_slot(const RoundArgs &a, const Run &r, int64_t w, int64_t c)
{
    const int sl = (c == udiv(first_elem(r, w), r.V)) ? 0 : 1;
    return a.partials + ((int64_t)(r.gw0 + w) * 2 + sl) * a.pstride;
}

// Target column c (position j = c mod (gamma+1) of lane ln) is done and
// its argmax is `arg` (the warp's lane 0 holds it).  Lane 0 writes the
// column's commit id and adds to the lane's ticket word, in one acq_rel
// atomic, 1 (bits 0-7: columns done) plus, for j < gamma, bit 8+j if
// draft j equals the argmax.  The completing column's warp reads every
// match bit from the word: the accept length is the run of set bits from
// bit 8, and it pads the commit ids after it with -1.
__device__ __noinline__ void verify_column_done(const RoundArgs &a, int64_t c, int32_t arg, int lane)
{
    const int gamma = a.gamma, gp1 = gamma + 1;
    const int64_t ln = udiv(c, gp1);
    const int j = (int)(c - ln * gp1);
    uint32_t word = 0;
    if (lane == 0) {
        const bool match = j < gamma && __ldg(a.drafts + ln * gamma + j) == arg;
        a.out_commit[ln * gp1 + j] = arg;
        const uint32_t add = 1u + ((match ? 1u : 0u) << (8 + j));
        word = atom_add_acq_rel(a.lane_ticket + ln, add) + add;
    }
    word = __shfl_sync(kFull, word, 0);
    if ((word & 0xFFu) != (uint32_t)gp1) return;
    const uint32_t flags = (word >> 8) & ((1u << gamma) - 1u);
    const int acc = __ffs(~flags) - 1 < gamma ? __ffs(~flags) - 1 : gamma;
    if (lane < gp1 && lane > acc) a.out_commit[ln * gp1 + lane] = -1;
    count_lane(a.counters, gamma, acc, lane);
    if (lane == 0) {
        a.out_accept[ln] = acc;
        a.lane_ticket[ln] = 0u;   // ready for the next launch
    }
}

// Sampled verify of target column c (position j = c mod (gamma+1) of lane
// ln) from its top-t_k list lst[0..n), best first -- speculative sampling
// with a one-hot draft ("A drafter inside the artifact", Ignis DFlash2
// page, "The numbers": sampled acceptance at T, top_p, top_k).  In float64
// and in list order: z_t = v_t / T; e_t = exp(z_t - z_0); S = sum e_t;
// p_t = e_t / S; the nucleus is the shortest prefix whose running sum of p
// reaches top_p; q_t = p_t / (that sum).  Draft j is accepted when u < q(draft)
// (u = uniforms[ln][j][0]); otherwise -- and always at position gamma, the
// bonus -- the token drawn is the first nucleus token (draft skipped) whose
// running q exceeds uniforms[ln][j][1] times the total q without the draft.
// Sums of doubles over the warp: the total in every lane, and the
// inclusive prefix (lane order) in each lane.
__device__ __forceinline__ double warp_sum_d(double v)
{
#pragma unroll
    for (int d = 16; d; d >>= 1) v += __shfl_xor_sync(kFull, v, d);
    return v;
}

__device__ __forceinline__ double warp_scan_d(double v, int lane)
{
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const double y = __shfl_up_sync(kFull, v, d);
        if (lane >= d) v += y;
    }
    return v;
}

__device__ __forceinline__ float warp_sum_f(float v)
{
#pragma unroll
    for (int d = 16; d; d >>= 1) v += __shfl_xor_sync(kFull, v, d);
    return v;
}

__device__ __forceinline__ float warp_scan_f(float v, int lane)
{
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const float y = __shfl_up_sync(kFull, v, d);
        if (lane >= d) v += y;
    }
    return v;
}

// The decisions of sampled_decide in float32, where each is certain.  Each
// term e_t = exp((v_t - v_0) / T) is computed with an absolute error below
// 3e-7 (the difference of two bf16 values, one multiplication by 1/T and
// expf each round once, and |x| e^x <= 1/e bounds what a relative error in
// the exponent does), so the probabilities p_t, their running sums and,
// with a nucleus sum of at least 1/4, the q_t and their running sums are
// off by less than 1e-4.  A decision whose float32 margin is at least 2e-4
// is therefore the one float64 takes.  Returns false -- nothing decided,
// float64 decides -- when a margin is smaller, the nucleus sum is below
// 1/4, or the list is longer than 32.
__device__ __forceinline__ bool sampled_decide_f32(const RoundArgs &a, const unsigned long long *lst, int n, int lane,
                                                   bool has_draft, int32_t draft, double u, double u2, bool &accepted,
                                                   int32_t &token)
{
    constexpr float kSure = 2e-4f;
    if (n > 32) return false;
    const float invT = (float)(1.0 / a.temperature);
    const bool h = lane < n;
    const unsigned long long e_ = h ? lst[lane] : 0ull;
    const float v0 = bf16_as_float(entry_raw(lst[0]));
    const float e = h ? expf((bf16_as_float(entry_raw(e_)) - v0) * invT) : 0.0f;
    const int32_t id = h ? (int32_t)entry_id(e_) : -1;
    const float p = e / warp_sum_f(e);
    const float cp = warp_scan_f(p, lane);
    const float top_p = (float)a.top_p;
    const uint32_t reach = __ballot_sync(kFull, h && cp >= top_p);
    const int last = reach ? __ffs(reach) - 1 : n - 1;
    // the nucleus cut: the running sum at it clears top_p (when it reaches
    // it at all) and the one before falls short of it, both by kSure
    const float c_last = __shfl_sync(kFull, cp, last);
    const float c_prev = __shfl_sync(kFull, cp, last > 0 ? last - 1 : 0);
    if (reach && c_last - top_p < kSure) return false;
    if (last > 0 && top_p - c_prev < kSure) return false;
    if (!(c_last >= 0.25f)) return false;   // also a NaN (a column topped by -Inf)
    const float q = lane <= last ? p / c_last : 0.0f;
    const uint32_t dm = __ballot_sync(kFull, lane <= last && id == draft && has_draft);
    const float qd = dm ? __shfl_sync(kFull, q, __ffs(dm) - 1) : 0.0f;
    if (has_draft && dm && fabs(u - (double)qd) < (double)kSure) return false;
    accepted = has_draft && u < (double)qd;
    if (accepted) {
        token = draft;
        return true;
    }
    // the draw: the first kept token (the draft skipped) whose running
    // weight exceeds u2 times the total
    const bool k = lane <= last && !(has_draft && id == draft);
    const float wgt = k ? q : 0.0f;
    const float target = (float)u2 * warp_sum_f(wgt);
    const float run = warp_scan_f(wgt, lane);
    const uint32_t x = __ballot_sync(kFull, k && run > target);
    if (!x) return false;
    const int pick = __ffs(x) - 1;
    const float r_pick = __shfl_sync(kFull, run, pick), r_prev = __shfl_sync(kFull, run - wgt, pick);
    if (r_pick - target < kSure || target - r_prev < kSure) return false;
    token = __shfl_sync(kFull, id, pick);
    return true;
}

// Returns whether the draft is accepted, and in token the position's token
// (the draft, or the draw), in every lane.  List entry t sits in lane t
// (t < 32) or lane t - 32.  The sums over the list are warp trees and the
// running sums warp scans, and p and q are products with one reciprocal:
// their rounding differs from sums in list order by about 1e-16 relative,
// so a decision can differ from one made in list order only within that
// distance of its boundary.  FP64 runs at a small fraction of the FP32
// rate on this GPU: about 80 double instructions per column instead of
// the 150 of four serial loops of broadcasts.
__device__ __noinline__ bool sampled_decide(const RoundArgs &a, int64_t c, const unsigned long long *lst, int n,
                                            int lane, int32_t &token_out)
{
    const int gamma = a.gamma, gp1 = gamma + 1;
    const int64_t ln = udiv(c, gp1);
    const int j = (int)(c - ln * gp1);
    const int32_t draft = j < gamma ? __ldg(a.drafts + ln * gamma + j) : -1;
    const double u = a.uniforms[(ln * gp1 + j) * 2], u2 = a.uniforms[(ln * gp1 + j) * 2 + 1];
    {
        bool acc32;
        int32_t tok32;
        if (sampled_decide_f32(a, lst, n, lane, j < gamma, draft, u, u2, acc32, tok32)) {
            token_out = tok32;
            return acc32;
        }
    }
    const double T = a.temperature;
    const bool ha = lane < n, hb = lane + 32 < n;
    const unsigned long long ea_ = ha ? lst[lane] : 0ull, eb_ = hb ? lst[lane + 32] : 0ull;
    const double z0 = (double)bf16_as_float(entry_raw(lst[0])) / T;
    const double ea = ha ? exp((double)bf16_as_float(entry_raw(ea_)) / T - z0) : 0.0;
    const double eb = hb ? exp((double)bf16_as_float(entry_raw(eb_)) / T - z0) : 0.0;
    const int32_t ida = ha ? (int32_t)entry_id(ea_) : -1, idb = hb ? (int32_t)entry_id(eb_) : -1;
    const double inv = 1.0 / warp_sum_d(ea + eb);
    const double pa = ea * inv, pb = eb * inv;
    // the nucleus: the shortest prefix whose running sum reaches top_p
    const double ca = warp_scan_d(pa, lane);
    const double cb = __shfl_sync(kFull, ca, 31) + warp_scan_d(pb, lane);
    const uint32_t ra = __ballot_sync(kFull, ha && ca >= a.top_p), rb = __ballot_sync(kFull, hb && cb >= a.top_p);
    int last;
    double C;
    if (ra) {
        last = __ffs(ra) - 1;
        C = __shfl_sync(kFull, ca, last);
    } else if (rb) {
        last = 32 + __ffs(rb) - 1;
        C = __shfl_sync(kFull, cb, last - 32);
    } else {
        last = n - 1;
        C = n > 32 ? __shfl_sync(kFull, cb, (n - 33) & 31) : __shfl_sync(kFull, ca, (n - 1) & 31);
    }
    const double invC = 1.0 / C;
    const double qa = lane <= last ? pa * invC : 0.0, qb = lane + 32 <= last ? pb * invC : 0.0;
    // q of the draft (0 outside the nucleus)
    const uint32_t da = __ballot_sync(kFull, lane <= last && ida == draft && draft >= 0);
    const uint32_t db = __ballot_sync(kFull, lane + 32 <= last && idb == draft && draft >= 0);
    double qd = 0.0;
    {
        const double xa = __shfl_sync(kFull, qa, da ? __ffs(da) - 1 : 0);
        const double xb = __shfl_sync(kFull, qb, db ? __ffs(db) - 1 : 0);
        qd = da ? xa : (db ? xb : 0.0);
    }
    const bool accepted = j < gamma && u < qd;
    int32_t token = draft;
    if (!accepted) {
        // a draw from q without the draft: the first kept token (list order,
        // the draft skipped) whose running weight exceeds u2 times the total
        const bool ka = lane <= last && ida != draft, kb = lane + 32 <= last && idb != draft;
        const double wa = ka ? qa : 0.0, wb = kb ? qb : 0.0;
        const double target = u2 * warp_sum_d(wa + wb);
        const double sa = warp_scan_d(wa, lane);
        const double sb = __shfl_sync(kFull, sa, 31) + warp_scan_d(wb, lane);
        const uint32_t xa = __ballot_sync(kFull, ka && sa > target), xb = __ballot_sync(kFull, kb && sb > target);
        const int32_t pa_id = __shfl_sync(kFull, ida, xa ? __ffs(xa) - 1 : 0);
        const int32_t pb_id = __shfl_sync(kFull, idb, xb ? __ffs(xb) - 1 : 0);
        // none exceeds it (rounding left the target at the very end): the last kept token
        const uint32_t la = __ballot_sync(kFull, ka), lb = __ballot_sync(kFull, kb);
        const int32_t last_a = __shfl_sync(kFull, ida, la ? 31 - __clz((int)la) : 0);
        const int32_t last_b = __shfl_sync(kFull, idb, lb ? 31 - __clz((int)lb) : 0);
        token = xa ? pa_id : xb ? pb_id : lb ? last_b : last_a;
    }
    token_out = token;
    return accepted;
}

// Sampled verify of target column c (as sampled_decide): the position's
// token goes to its commit id and its acceptance bit to the lane's ticket
// word, as in verify_column_done.
__device__ __noinline__ void sampled_column_done(const RoundArgs &a, int64_t c, const unsigned long long *lst, int n,
                                                 int lane)
{
    const int gamma = a.gamma, gp1 = gamma + 1;
    const int64_t ln = udiv(c, gp1);
    const int j = (int)(c - ln * gp1);
    int32_t token;
    const bool accepted = sampled_decide(a, c, lst, n, lane, token);
    uint32_t word = 0;
    if (lane == 0) {
        a.out_commit[ln * gp1 + j] = token;
        const uint32_t add = 1u + ((accepted ? 1u : 0u) << (8 + j));
        word = atom_add_acq_rel(a.lane_ticket + ln, add) + add;
    }
    word = __shfl_sync(kFull, word, 0);
    if ((word & 0xFFu) != (uint32_t)gp1) return;
    const uint32_t flags = (word >> 8) & ((1u << gamma) - 1u);
    const int acc = __ffs(~flags) - 1 < gamma ? __ffs(~flags) - 1 : gamma;
    if (lane < gp1 && lane > acc) a.out_commit[ln * gp1 + lane] = -1;
    count_lane(a.counters, gamma, acc, lane);
    if (lane == 0) {
        a.out_accept[ln] = acc;
        a.lane_ticket[ln] = 0u;   // ready for the next launch
    }
}

// Diagnostic of the bounded waits: one thread waits on an mbarrier that
// nothing arrives on (limit limit_ns), then once more on the same phase; the
// first wait must give up and flag, the second return at once.  Writes the
// two results and their durations to out[0..3].
__global__ void wait_timeout_probe(uint64_t limit_ns, unsigned long long *out)
{
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    s_gave_up = 0u;
    mbar_init(&bar, 1);
    fence_mbar_init();
    const uint64_t t0 = global_ns();
    const bool first = mbar_wait(&bar, 0, limit_ns);
    const uint64_t t1 = global_ns();
    const bool second = mbar_wait(&bar, 0, limit_ns);
    const uint64_t t2 = global_ns();
    out[0] = first;
    out[1] = t1 - t0;
    out[2] = second;
    out[3] = t2 - t1;
}

}  // namespace
