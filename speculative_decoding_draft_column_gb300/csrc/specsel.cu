// libspecsel: exact per-column top-k and fused greedy verify over bf16 logits
// for one GB300 (sm_103a).
//
// The operations ("A drafter inside the artifact", Ignis DFlash2 page,
// section "How it works"):
//   * top-k over each draft column of V logits: largest first, ties to the
//     smaller token id (third paragraph);
//   * greedy verify: per target column the argmax (same tie rule), then per
//     lane the longest run of drafts equal to those argmaxes, committed
//     together with the target's own next token (first paragraph).
//
// Design (one streaming pass over the logits, no tensor cores -- the step is
// a pure reduction bound by HBM bandwidth):
//   * Every warp of a full-GPU grid (16 warps per CTA, one CTA per SM) owns a
//     contiguous slice of the flat run of logits (draft columns one after the
//     other, then target columns), the same number of 16-byte vectors for
//     every warp.  A slice may start or end inside a column.  The warps never
//     wait on one another in the streaming loop.
//   * Each warp streams its slice through its own ring of three 4 KiB stages
//     in shared memory, filled by one-dimensional bulk copies
//     (cp.async.bulk, completion on an mbarrier); lane 0 refills a stage as
//     soon as the warp is done with it, so 12 KiB per warp (192 KiB per SM)
//     stay in flight.
//   * Per column segment the warp keeps a candidate buffer in shared memory:
//     packed (value key, id, bits) entries appended in increasing id order.
//     A stage is skipped after one bf16x2 max tree per lane and one compare
//     against the column's threshold.  The threshold is a certificate: a key
//     that kk elements already reach.  It is seeded from the first stage
//     (the kk-th largest of the lane maxima) and tightened by pruning the
//     buffer to its kk best (a bisection over the 16 key bits); since the warp
//     meets elements in id order, a later element equal to the threshold is
//     worse than every kept entry and is rejected (strict filter).
//   * A column seen whole by one warp is emitted by it.  Otherwise every warp
//     that saw part of it publishes its kk best (and their certificate) to
//     scratch and takes the column's ticket; the warp that completes the
//     column merges the lists in slice order -- the logits are read once.
//   * Verify columns are the k = 1 instance; the warp that completes the last
//     of a lane's gamma+1 columns runs the prefix match (one lane per
//     position).  Tickets are reset by their last user, so launches replay.
//   * Masked elements (past a column or the buffer) are bf16 NaN: bf16 max
//     ignores them, ordered compares reject them.  The buffer's ragged first
//     and last 16-byte vectors are read element by element, so no load or
//     copy touches memory outside the caller's buffer.
//   * Every mbarrier wait is bounded in time; a wait that gives up sets a flag
//     (spec_device_status) and the kernel still ends.

#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <string>

#include "specsel.h"

namespace {

constexpr int kWarpsPerCta = 16;
constexpr int kThreads = kWarpsPerCta * 32;
constexpr int kStageVec = 256;                     // 16-byte vectors per warp stage (4 KiB)
constexpr int kLaneVec = kStageVec / 32;           // vectors per lane per stage
constexpr int kStages = 3;                         // per-warp ring depth (12 KiB in flight per warp)
constexpr int kBufCap = 128;                       // per-warp candidate buffer (entries)
constexpr int kMinSliceVec = 2 * kStageVec;        // smallest slice a warp is given
constexpr uint64_t kWaitLimitNs = 4000000000ull;   // bound on any mbarrier wait: 4 s of wall time
constexpr unsigned kFull = 0xffffffffu;
constexpr uint32_t kNaN2 = 0x7FFF7FFFu;            // two bf16 NaNs: the mask value

static_assert(kBufCap >= 2 * SPEC_MAX_K && kBufCap % 32 == 0, "a pruned buffer must leave room");

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
    // warps [0, d_warps) stream the draft logits, [d_warps, d_warps + t_warps) the target logits
    int32_t d_warps, t_warps;
    // scratch
    unsigned long long *partials;   // [(d_warps + t_warps) * 2][pstride = k + 2]
    unsigned int *col_ticket;       // [d_cols + t_cols]
    unsigned int *col_cert;         // [d_cols + t_cols]: best certified key published for a split column
    unsigned int *lane_ticket;      // [lanes]
    int32_t *t_argmax;              // [t_cols]
    int32_t pstride;
};

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

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(smem_u32(bar)), "r"(parity)
                 : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase with the given parity to complete, for at most
// kWaitLimitNs of wall time; on giving up, flag the error and report false
// (the data is then garbage, but the kernel still terminates).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > kWaitLimitNs) {
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

// ---- candidate buffers ------------------------------------------------------

struct Pruned {
    int n;       // entries kept (kk)
    uint32_t t;  // their certificate: the kk-th largest key
};

// Prune the warp buffer wb[0..n) (n >= kk, any order) to its kk best
// entries; returns kk and the kk-th largest key t (kk entries reach it: a
// certificate).  Ties at t go to the smallest ids (token ids, or mapped
// vocabulary ids for a shortlist), found by a bisection over the id bits only
// when there are more ties than places.
__device__ __noinline__ Pruned buf_prune(unsigned long long *wb, int n, int kk, int lane)
{
    constexpr int Q = kBufCap / 32;
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

struct ColState {
    int n;          // entries in the buffer
    uint32_t own;   // own certified key (last prune)
    uint32_t cert;  // certificate from elsewhere (seed or merge), inclusive
    bool open;      // the warp has started this column
    int seen;       // elements of the column this warp has scanned (saturating)
};

// ---- the per-warp stream ------------------------------------------------------

// Shared memory of one warp: its copy ring, candidate buffer and barriers.
struct WarpSmem {
    uint4 ring[kStages][kStageVec];
    unsigned long long buf[kBufCap];
    uint64_t full[kStages];
};

constexpr size_t kSmemBytes = (size_t)kWarpsPerCta * sizeof(WarpSmem);

// One buffer (draft or target logits) seen as a flat run of N = cols * V
// elements on the 16-byte vector grid: vector j holds elements
// [8j - mis, 8j - mis + 8).  The run is cut into W slices of whole vectors;
// slice w = vectors [start(w), start(w+1)), start(w) = floor(w * NV / W).
struct Run {
    const uint16_t *buf;
    const uint4 *vb;          // 16-byte aligned base, at or just below buf
    int64_t V, N, NV;
    int64_t jlo, jhi;         // vectors [jlo, jhi) lie wholly inside the buffer
    int W, gw0;               // warps on this run; global index of its slice 0
    int kk;
    int mis;
    bool draft;
};

__device__ __forceinline__ int64_t slice_start(const Run &r, int64_t w) { return w * r.NV / r.W; }
__device__ __forceinline__ int64_t owner(const Run &r, int64_t j) { return ((j + 1) * r.W - 1) / r.NV; }
__device__ __forceinline__ int64_t first_elem(const Run &r, int64_t w)
{
    const int64_t g = 8 * slice_start(r, w) - r.mis;
    return g > 0 ? g : 0;
}

// The list slot of warp w for column c: 0 if c is the first column of the
// slice, else 1 (a slice holds part of at most two columns).
__device__ __forceinline__ unsigned long long *list_slot(const RoundArgs &a, const Run &r, int64_t w, int64_t c)
{
    const int sl = (c == first_elem(r, w) / r.V) ? 0 : 1;
    return a.partials + ((int64_t)(r.gw0 + w) * 2 + sl) * a.pstride;
}

// Write a finished column: its best entries (in the buffer, id order) are
// ranked by value; top-k outputs, or for a target column the argmax and, for
// the lane's last column, the prefix match (one lane per position).
__device__ __noinline__ void emit_column(const RoundArgs &a, const Run &r, int64_t c,
                                         const unsigned long long *wb, int n, int lane)
{
    const int kk = r.kk;
    for (int i = lane; i < n; i += 32) {
        const unsigned long long e = wb[i];
        int rank = 0;
        for (int j = 0; j < n; ++j) rank += wb[j] > e;
        if (r.draft) {
            a.out_vals[c * kk + rank] = entry_raw(e);
            a.out_ids[c * kk + rank] = (int32_t)entry_id(e);
        } else if (rank == 0) {
            a.t_argmax[c] = (int32_t)entry_id(e);
        }
    }
    if (r.draft) return;
    const int gp1 = a.gamma + 1;
    const int64_t ln = c / gp1;
    __threadfence();
    __syncwarp();
    unsigned last = 0;
    if (lane == 0) last = atomicAdd(a.lane_ticket + ln, 1u) == (unsigned)a.gamma;
    if (!__shfl_sync(kFull, last, 0)) return;
    __threadfence();
    const int32_t tj = lane < gp1 ? __ldcg(a.t_argmax + ln * gp1 + lane) : 0;
    const int32_t dj = lane < a.gamma ? __ldg(a.drafts + ln * a.gamma + lane) : 0;
    const uint32_t miss = __ballot_sync(kFull, lane < a.gamma && dj != tj);
    const int acc = miss ? __ffs(miss) - 1 : a.gamma;
    if (lane < gp1) a.out_commit[ln * gp1 + lane] = lane <= acc ? tj : -1;
    if (lane == 0) {
        a.out_accept[ln] = acc;
        a.lane_ticket[ln] = 0u;   // ready for the next launch
    }
}

// Column c's segment in this warp is over.  If the warp saw the whole column,
// emit it; otherwise publish the warp's list and take the column's ticket;
// the warp that completes the column merges every warp's list (in slice
// order, hence in id order) and emits it.
template <bool MAPPED>
__device__ __noinline__ void finish_column(const RoundArgs &a, const Run &r, int w, int64_t c,
                                           unsigned long long *wb, int n_in, uint32_t own_in, int lane)
{
    ColState cs = {n_in, own_in, 0u, true, 0};
    const int kk = r.kk;
    if (cs.n > kk) { const Pruned pq = buf_prune(wb, cs.n, kk, lane); cs.n = pq.n; cs.own = pq.t; }
    const int64_t wf = owner(r, (c * r.V + r.mis) >> 3);
    const int64_t wl = owner(r, ((c + 1) * r.V - 1 + r.mis) >> 3);
    if (wf == wl) {
        emit_column(a, r, c, wb, cs.n, lane);
        return;
    }
    // publish: the list (kk entries, id order, 0-padded), in slot kk its
    // certificate -- the smallest key of a full list (kk entries reach it) --
    // and in slot kk + 1 its length
    uint32_t mk = 0xFFFFFFFFu;
    for (int i = lane; i < cs.n; i += 32) {
        const uint32_t ky = entry_key(wb[i]);
        mk = ky < mk ? ky : mk;
    }
    mk = __reduce_min_sync(kFull, mk);
    unsigned long long *mine = list_slot(a, r, w, c);
    for (int i = lane; i < cs.n; i += 32) mine[i] = wb[i];
    if (lane == 0) {
        mine[kk] = cs.n == kk ? mk : 0u;
        mine[kk + 1] = (unsigned long long)cs.n;
    }
    __threadfence();
    __syncwarp();
    const int64_t tix = r.draft ? c : a.d_cols + c;
    unsigned last = 0;
    if (lane == 0) last = atomicAdd(a.col_ticket + tix, 1u) == (unsigned)(wl - wf);
    if (!__shfl_sync(kFull, last, 0)) return;
    __threadfence();
    // merge.  The best certificate (the column's shared one, or any full
    // list's) bounds the column's kk-th key; only entries at or above it are
    // gathered, list by list in slice order (hence id order), each lane
    // loading one list, all lists in flight at once.
    cs.n = 0;
    cs.own = 0;
    cs.cert = ld_relaxed(a.col_cert + tix);
    const int64_t nparts = wl - wf + 1;
    for (int64_t q0 = 0; q0 < nparts; q0 += 32) {
        uint32_t key = 0;
        if (q0 + lane < nparts) key = (uint32_t)__ldcg(list_slot(a, r, wf + q0 + lane, c) + kk);
        key = __reduce_max_sync(kFull, key);
        cs.cert = key > cs.cert ? key : cs.cert;
    }
    for (int64_t q0 = 0; q0 < nparts; q0 += 32) {
        const bool mine_l = q0 + lane < nparts;
        const unsigned long long *lst = mine_l ? list_slot(a, r, wf + q0 + lane, c) : nullptr;
        const int len = mine_l ? (int)__ldcg(lst + kk + 1) : 0;
        const int maxlen = __reduce_max_sync(kFull, len);
        for (int i0 = 0; i0 < maxlen; i0 += 8) {
            unsigned long long e8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) e8[i] = i0 + i < len ? __ldcg(lst + i0 + i) : 0ull;
            uint32_t ok = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) ok |= (uint32_t)(e8[i] != 0ull && entry_key(e8[i]) >= cs.cert) << i;
            for (;;) {
                int total;
                const int excl = warp_exclusive_sum(__popc(ok), lane, total);
                if (total == 0) break;
                const int space = kBufCap - cs.n;
                int pos = excl;
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if ((ok >> i) & 1u) {
                        if (pos < space) {
                            wb[cs.n + pos] = e8[i];
                            ok &= ~(1u << i);
                        }
                        ++pos;
                    }
                __syncwarp();
                if (total <= space) {
                    cs.n += total;
                    break;
                }
                const Pruned pq = buf_prune(wb, kBufCap, kk, lane);
                cs.n = pq.n;
                cs.own = pq.t;
                if (cs.own > cs.cert) cs.cert = cs.own;
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (entry_key(e8[i]) < cs.cert) ok &= ~(1u << i);
            }
        }
    }
    if (cs.n > kk) { const Pruned pq = buf_prune(wb, cs.n, kk, lane); cs.n = pq.n; cs.own = pq.t; }
    emit_column(a, r, c, wb, cs.n, lane);
    if (lane == 0) {
        a.col_ticket[tix] = 0u;   // ready for the next launch
        a.col_cert[tix] = 0u;
    }
}

// Issue the bulk copy of stage i of slice [J0, J1) into ring slot i % kStages.
// Only vectors wholly inside the buffer are copied; the (at most two) edge
// vectors of the buffer are read element by element by the consumer.
__device__ __forceinline__ void issue_stage(const Run &r, WarpSmem &ws, int64_t J0, int64_t J1, int64_t i)
{
    const int st = (int)(i % kStages);
    const int64_t vs = J0 + i * kStageVec;
    const int64_t ve = vs + kStageVec < J1 ? vs + kStageVec : J1;
    const int64_t is = vs > r.jlo ? vs : r.jlo;
    const int64_t ie = ve < r.jhi ? ve : r.jhi;
    const uint32_t bytes = ie > is ? (uint32_t)((ie - is) * 16) : 0u;
    fence_proxy_async();
    mbar_arrive_expect_tx(&ws.full[st], bytes);
    if (bytes) bulk_g2s(&ws.ring[st][is - vs], r.vb + is, bytes, &ws.full[st]);
}

// One warp streams its slice w of run r: every column segment gets a
// candidate buffer and a threshold; finished columns are emitted or merged.
template <int SLOTS, bool MAPPED>
__device__ __forceinline__ void stream_slice(const RoundArgs &a, const Run &r, int w,
                                             const int32_t *__restrict__ id_map, WarpSmem &ws, int lane)
{
    const int64_t J0 = slice_start(r, w), J1 = slice_start(r, w + 1);
    if (J1 <= J0) return;
    const int64_t nst = (J1 - J0 + kStageVec - 1) / kStageVec;
    const int kk = r.kk;
    unsigned long long *wb = ws.buf;
    if (lane == 0)
        for (int64_t i = 0; i < nst && i < kStages; ++i) issue_stage(r, ws, J0, J1, i);

    int64_t c = first_elem(r, w) / r.V;       // current column
    ColState cs = {0, 0u, 0u, false, 0};
    // a column split across warps has a shared certificate in global memory:
    // every warp raises it with its own certified keys and filters against
    // it (read one stage late, so the load latency hides behind the stream)
    bool shared = false;
    int64_t tix = 0;
    uint32_t gcert = 0;

    for (int64_t i = 0; i < nst; ++i) {
        const int st = (int)(i % kStages);
        mbar_wait(&ws.full[st], (uint32_t)(i / kStages) & 1u);
        const int64_t vs = J0 + i * kStageVec;
        const int64_t ve = vs + kStageVec < J1 ? vs + kStageVec : J1;
        const int64_t g_first = 8 * vs - r.mis > 0 ? 8 * vs - r.mis : 0;
        const int64_t g_end = 8 * ve - r.mis < r.N ? 8 * ve - r.mis : r.N;   // exclusive
        for (;;) {
            // the part of column c inside this stage, elements outside as NaN
            const int64_t cb = c * r.V, ce = cb + r.V;
            const bool whole = cb <= g_first && ce >= g_end;
            uint4 y[kLaneVec];
            if (whole && ve - vs == kStageVec && vs >= r.jlo && ve <= r.jhi) {
                // the common case: a full stage, inside one column, no buffer edge
                const uint4 *src = &ws.ring[st][lane];
#pragma unroll
                for (int u = 0; u < kLaneVec; ++u) y[u] = src[u * 32];
            } else {
#pragma unroll
                for (int u = 0; u < kLaneVec; ++u) {
                    const int64_t j = vs + u * 32 + lane;
                    if (j >= ve) y[u] = make_uint4(kNaN2, kNaN2, kNaN2, kNaN2);
                    else if (j < r.jlo || j >= r.jhi) {
                        y[u] = load_edge(r.buf, j, r.mis, cb, ce < r.N ? ce : r.N);
                        ws.ring[st][j - vs] = y[u];   // edge vectors are not copied in: keep them here
                    }
                    else y[u] = ws.ring[st][j - vs];
                    if (!whole) {
                        const int64_t g0 = 8 * j - r.mis;
                        uint32_t wv[4] = {y[u].x, y[u].y, y[u].z, y[u].w};
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            const int64_t ga = g0 + 2 * h;
                            if (ga < cb || ga >= ce) wv[h] = (wv[h] & 0xFFFF0000u) | 0x7FFFu;
                            if (ga + 1 < cb || ga + 1 >= ce) wv[h] = (wv[h] & 0x0000FFFFu) | 0x7FFF0000u;
                        }
                        y[u] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                    }
                }
            }

            if (!cs.open) {
                cs.open = true;
                shared = owner(r, (c * r.V + r.mis) >> 3) != owner(r, ((c + 1) * r.V - 1 + r.mis) >> 3);
                tix = r.draft ? c : a.d_cols + c;
                gcert = 0;
            }
            if (gcert > cs.cert) cs.cert = gcert;
            if (cs.seen < 8 * kStageVec) {
                // seed, until the warp has seen a full stage of the column: the
                // kk-th largest of the group maxima certifies kk elements
                constexpr int G = (SLOTS == 1) ? 1 : 4;
                constexpr int PER = kLaneVec / G;
                uint32_t key[G];
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    uint32_t m = vmax(y[g * PER]);
#pragma unroll
                    for (int u = 1; u < PER; ++u) m = bmax2(m, vmax(y[g * PER + u]));
                    key[g] = order_key(hmax_splat(m) & 0xFFFFu);
                }
                uint32_t seed = 0;
                if (kk == 1) {
                    seed = __reduce_max_sync(kFull, key[0]);
                } else {
#pragma unroll 1
                    for (int bit = 15; bit >= 0; --bit) {
                        const uint32_t tr = seed | (1u << bit);
                        int cnt = 0;
#pragma unroll
                        for (int g = 0; g < G; ++g) cnt += __popc(__ballot_sync(kFull, key[g] >= tr));
                        if (cnt >= kk) seed = tr;
                    }
                }
                cs.cert = seed > cs.cert ? seed : cs.cert;
                if (shared && lane == 0 && seed > gcert) atomicMax(a.col_cert + tix, seed);
                const int64_t lo = cb > g_first ? cb : g_first, hi = ce < g_end ? ce : g_end;
                cs.seen += (int)(hi - lo);
            }
            Filter f = make_filter(cs.own, cs.cert, MAPPED);
            uint32_t m = vmax(y[0]);
#pragma unroll
            for (int u = 1; u < kLaneVec; ++u) m = bmax2(m, vmax(y[u]));
            const bool pass = f.strict ? any_gt(m, f.thr2) : any_ge(m, f.thr2);
            if (__ballot_sync(kFull, pass)) {
                // append the candidates: one warp prefix sum gives every lane
                // its places, each lane writes its own (their order in the
                // buffer does not matter, ties are settled by id when pruning)
                const int64_t id_lane = 8 * (vs + lane) - r.mis - cb;   // id of element 0, vector 0
                const uint16_t *sv = reinterpret_cast<const uint16_t *>(&ws.ring[st][0]);
                uint64_t bits = 0;   // this lane's candidates: bit 8u+e = element e of vector u
#pragma unroll
                for (int u = 0; u < kLaneVec; ++u)
                    if (pass && (f.strict ? any_gt(vmax(y[u]), f.thr2) : any_ge(vmax(y[u]), f.thr2)))
                        bits |= (uint64_t)elem_mask(y[u], f) << (8 * u);
                for (;;) {
                    int total;
                    const int excl = warp_exclusive_sum(__popcll(bits), lane, total);
                    if (total == 0) break;
                    const int space = kBufCap - cs.n;
                    int pos = excl;
                    uint64_t rest = bits;
                    while (rest && pos < space) {
                        const int b = __ffsll((long long)rest) - 1;
                        rest &= rest - 1;
                        const int u = b >> 3, e = b & 7;
                        uint32_t cid = (uint32_t)(id_lane + 256 * u + e);
                        if (MAPPED) cid = (uint32_t)__ldg(id_map + cid);
                        wb[cs.n + pos] = pack_entry(bf16_as_float(sv[8 * (u * 32 + lane) + e]), cid);
                        ++pos;
                    }
                    __syncwarp();
                    if (total <= space) {
                        cs.n += total;
                        break;
                    }
                    // the buffer is full: prune it, then keep only what still
                    // reaches the new key (inclusively: the rest of this
                    // stage may hold smaller ids than entries just kept)
                    const Pruned pq = buf_prune(wb, kBufCap, kk, lane);
                    cs.n = pq.n;
                    cs.own = pq.t;
                    const float tv = bf16_as_float(key_to_raw(cs.own));
                    uint64_t keep = 0;
                    for (uint64_t q = rest; q; q &= q - 1) {
                        const int b = __ffsll((long long)q) - 1;
                        if (bf16_as_float(sv[8 * ((b >> 3) * 32 + lane) + (b & 7)]) >= tv) keep |= 1ull << b;
                    }
                    bits = keep;
                }
                __syncwarp();
                // a first threshold as soon as kk candidates are in; after
                // that, prune only when the buffer is three-quarters full (an
                // append is cheap, a prune is a 16-step bisection)
                if (cs.n >= kk && (cs.own == 0 || cs.n >= kBufCap * 3 / 4)) {
                    const Pruned pq = buf_prune(wb, cs.n, kk, lane);
                    cs.n = pq.n;
                    cs.own = pq.t;
                    if (shared && lane == 0 && cs.own > cs.cert) atomicMax(a.col_cert + tix, cs.own);
                }
            }

            if (ce > g_end) break;                    // column c goes on past this stage
            finish_column<MAPPED>(a, r, w, c, wb, cs.n, cs.own, lane);
            cs = {0, 0u, 0u, false, 0};
            ++c;
            if (c * r.V >= g_end) break;              // next column starts in a later stage
        }
        __syncwarp();                                  // every lane is done with the slot
        if (lane == 0 && i + kStages < nst) issue_stage(r, ws, J0, J1, i + kStages);
        if (cs.open && shared) gcert = ld_relaxed(a.col_cert + tix);
    }
    // the slice ended inside column c: publish what this warp saw of it
    if (cs.open) finish_column<MAPPED>(a, r, w, c, wb, cs.n, cs.own, lane);
}

template <int SLOTS, bool MAPPED>
__global__ void __launch_bounds__(kThreads, 1) spec_round_kernel(const __grid_constant__ RoundArgs a)
{
    extern __shared__ __align__(128) unsigned char smem[];
    const int lane = threadIdx.x & 31;
    const int gw = blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
    WarpSmem &ws = reinterpret_cast<WarpSmem *>(smem)[threadIdx.x >> 5];
    if (gw >= a.d_warps + a.t_warps) return;
    if (lane == 0) {
        for (int st = 0; st < kStages; ++st) mbar_init(&ws.full[st], 1);
        fence_mbar_init();
    }
    __syncwarp();

    Run r;
    const bool draft = gw < a.d_warps;
    r.draft = draft;
    r.buf = draft ? a.draft : a.target;
    r.V = draft ? a.d_V : a.t_V;
    r.N = (draft ? a.d_cols : a.t_cols) * r.V;
    r.W = draft ? a.d_warps : a.t_warps;
    r.gw0 = draft ? 0 : a.d_warps;
    r.kk = draft ? a.k : 1;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(r.buf);
    r.mis = (int)((a0 >> 1) & 7);                       // element phase of buf in 16 B
    r.vb = reinterpret_cast<const uint4 *>(a0 - 2 * (uintptr_t)r.mis);
    r.NV = (r.N + r.mis + 7) >> 3;
    r.jlo = r.mis ? 1 : 0;
    r.jhi = ((r.N + r.mis) & 7) ? r.NV - 1 : r.NV;
    if (r.jhi < r.jlo) r.jhi = r.jlo;
    const int w = gw - r.gw0;
    if (draft) stream_slice<SLOTS, MAPPED>(a, r, w, a.id_map, ws, lane);
    else stream_slice<1, false>(a, r, w, nullptr, ws, lane);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool init = false;
    int sms = 0;
    int occ[2][2] = {{0, 0}, {0, 0}};   // resident CTAs per SM, [slots-1][mapped]
    // Scratch: [col tickets | lane tickets | target argmax | partial lists].
    // Each region keeps its place and capacity until the whole area is
    // reallocated (and zeroed), so a ticket is never laid over stale data.
    void *scratch = nullptr;
    size_t scratch_bytes = 0;
    int64_t cap_cols = 0, cap_lanes = 0, cap_tcols = 0, cap_part = 0;
    void *staging = nullptr;
    size_t staging_bytes = 0;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
std::atomic<int64_t> g_launches{0};
thread_local cudaStream_t t_stream = nullptr;
thread_local std::string t_err;

spec_status fail(spec_status st, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
spec_status fail(spec_status st, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_err = buf;
    return st;
}

spec_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(SPEC_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

template <int S, bool M>
void *kernel_ptr() { return reinterpret_cast<void *>(spec_round_kernel<S, M>); }

spec_status device_state(DeviceState **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(SPEC_ERR_CUDA, "device ordinal %d unsupported", dev);
    DeviceState &d = g_dev[dev];
    if (!d.init) {
        e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        void *kp[2][2] = {{kernel_ptr<1, false>(), kernel_ptr<1, true>()},
                          {kernel_ptr<2, false>(), kernel_ptr<2, true>()}};
        for (int s = 0; s < 2; ++s)
            for (int m = 0; m < 2; ++m) {
                e = cudaFuncSetAttribute(kp[s][m], cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
                if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
                e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.occ[s][m], kp[s][m], kThreads, kSmemBytes);
                if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
                if (d.occ[s][m] < 1) d.occ[s][m] = 1;
            }
        d.init = true;
    }
    *out = &d;
    return SPEC_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct ScratchPtrs {
    unsigned int *col_ticket;
    unsigned int *lane_ticket;
    int32_t *t_argmax;
    unsigned long long *partials;
};

struct ScratchCaps {
    int64_t cols, lanes, tcols, part;   // part = partial-list entries (u64)
};

size_t scratch_bytes(const ScratchCaps &c)
{
    return align256((size_t)c.cols * 4) + align256((size_t)c.lanes * 4) + align256((size_t)c.tcols * 4) +
           align256((size_t)c.part * 8);
}

ScratchPtrs scratch_ptrs(const DeviceState &d)
{
    char *p = static_cast<char *>(d.scratch);
    ScratchPtrs s;
    s.col_ticket = reinterpret_cast<unsigned int *>(p);
    p += align256((size_t)d.cap_cols * 4);
    s.lane_ticket = reinterpret_cast<unsigned int *>(p);
    p += align256((size_t)d.cap_lanes * 4);
    s.t_argmax = reinterpret_cast<int32_t *>(p);
    p += align256((size_t)d.cap_tcols * 4);
    s.partials = reinterpret_cast<unsigned long long *>(p);
    return s;
}

bool stream_capturing(cudaStream_t st)
{
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return false;
    return cs != cudaStreamCaptureStatusNone;
}

// Grow (never shrink) the device's scratch so that every region covers
// `need`; fresh scratch is zeroed, and the kernels leave every ticket at zero
// when they finish.
spec_status ensure_scratch(DeviceState &d, const ScratchCaps &need, cudaStream_t st)
{
    if (d.scratch && need.cols <= d.cap_cols && need.lanes <= d.cap_lanes && need.tcols <= d.cap_tcols &&
        need.part <= d.cap_part)
        return SPEC_OK;
    if (stream_capturing(st))
        return fail(SPEC_ERR_ALLOC, "scratch must grow during stream capture; call spec_reserve before capturing");
    auto grow = [](int64_t have, int64_t want) { return want <= have ? have : want + want / 4 + 64; };
    ScratchCaps c;
    c.cols = grow(d.cap_cols, need.cols);
    c.lanes = grow(d.cap_lanes, need.lanes);
    c.tcols = grow(d.cap_tcols, need.tcols);
    c.part = grow(d.cap_part, need.part);
    const size_t bytes = scratch_bytes(c);
    cudaError_t e;
    if (d.scratch) {
        e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
        cudaFree(d.scratch);
        d.scratch = nullptr;
        d.scratch_bytes = 0;
        d.cap_cols = d.cap_lanes = d.cap_tcols = d.cap_part = 0;
    }
    e = cudaMalloc(&d.scratch, bytes);
    if (e != cudaSuccess) {
        d.scratch = nullptr;
        cudaGetLastError();
        return fail(SPEC_ERR_ALLOC, "cudaMalloc(%zu) for scratch: %s", bytes, cudaGetErrorString(e));
    }
    e = cudaMemset(d.scratch, 0, bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset scratch");
    d.scratch_bytes = bytes;
    d.cap_cols = c.cols;
    d.cap_lanes = c.lanes;
    d.cap_tcols = c.tcols;
    d.cap_part = c.part;
    return SPEC_OK;
}

int64_t vectors_of(const void *buf, int64_t n_elems)
{
    const int64_t mis = (int64_t)((reinterpret_cast<uintptr_t>(buf) >> 1) & 7);
    return (n_elems + mis + 7) >> 3;
}

// Split the warps of a full-GPU grid between the draft and the target logits
// in proportion to their 16-byte vectors, so that every warp streams the same
// number of bytes.  No slice is made smaller than kMinSliceVec vectors, and
// the published lists (two per warp, kk_stride entries each) must fit in
// max_partials entries.
void split_warps(int64_t nv_d, int64_t nv_t, int64_t max_warps, int kk_stride, int64_t max_partials,
                 int32_t *w_d, int32_t *w_t)
{
    int64_t total = max_warps;
    const int64_t cap = max_partials / (2 * (int64_t)kk_stride);
    if (total > cap) total = cap;
    if (total < 2) total = 2;
    auto limit = [](int64_t nv) { const int64_t m = nv / kMinSliceVec; return m < 1 ? (int64_t)1 : m; };
    int64_t d = 0, t = 0;
    if (nv_d > 0 && nv_t > 0) {
        d = (int64_t)((double)total * (double)nv_d / (double)(nv_d + nv_t) + 0.5);
        if (d < 1) d = 1;
        if (d > total - 1) d = total - 1;
        t = total - d;
    } else if (nv_d > 0) {
        d = total;
    } else {
        t = total;
    }
    if (nv_d > 0 && d > limit(nv_d)) d = limit(nv_d);
    if (nv_t > 0 && t > limit(nv_t)) t = limit(nv_t);
    *w_d = (int32_t)d;
    *w_t = (int32_t)t;
}

bool misaligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; }

spec_status check_topk_args(const uint16_t *logits, int64_t cols, int64_t V, int32_t k, const void *vals,
                            const void *ids)
{
    if (cols < 0) return fail(SPEC_ERR_ARG, "cols = %lld < 0", (long long)cols);
    if (V < 1 || V > INT32_MAX) return fail(SPEC_ERR_ARG, "V = %lld outside [1, 2^31-1]", (long long)V);
    if (k < 1 || k > SPEC_MAX_K || (int64_t)k > V)
        return fail(SPEC_ERR_ARG, "k = %d outside [1, min(V, %d)]", k, SPEC_MAX_K);
    if (cols == 0) return SPEC_OK;
    if (!logits || !vals || !ids) return fail(SPEC_ERR_ARG, "null pointer");
    if (misaligned(logits, 2) || misaligned(vals, 2) || misaligned(ids, 4))
        return fail(SPEC_ERR_ARG, "misaligned pointer (logits/out_vals need 2 bytes, out_ids 4)");
    if (cols > INT64_MAX / V) return fail(SPEC_ERR_ARG, "cols * V overflows");
    return SPEC_OK;
}

spec_status check_verify_args(const uint16_t *tl, const int32_t *drafts, int64_t lanes, int32_t gamma,
                              int64_t V, const int32_t *acc, const int32_t *com)
{
    if (lanes < 0) return fail(SPEC_ERR_ARG, "lanes = %lld < 0", (long long)lanes);
    if (gamma < 1 || gamma > SPEC_MAX_GAMMA)
        return fail(SPEC_ERR_ARG, "gamma = %d outside [1, %d]", gamma, SPEC_MAX_GAMMA);
    if (V < 1 || V > INT32_MAX) return fail(SPEC_ERR_ARG, "V = %lld outside [1, 2^31-1]", (long long)V);
    if (lanes == 0) return SPEC_OK;
    if (!tl || !drafts || !acc || !com) return fail(SPEC_ERR_ARG, "null pointer");
    if (misaligned(tl, 2) || misaligned(drafts, 4) || misaligned(acc, 4) || misaligned(com, 4))
        return fail(SPEC_ERR_ARG, "misaligned pointer");
    if (lanes > INT64_MAX / ((int64_t)(gamma + 1) * V)) return fail(SPEC_ERR_ARG, "lanes * (gamma+1) * V overflows");
    return SPEC_OK;
}

// Plan and launch one kernel covering a top-k part and/or a verify part.
spec_status launch_round(const uint16_t *draft, int64_t cols, int64_t V, int32_t k, const int32_t *id_map,
                         uint16_t *vals, int32_t *ids, const uint16_t *target, const int32_t *drafts,
                         int64_t lanes, int32_t gamma, int64_t tV, int32_t *acc, int32_t *com)
{
    if (cols == 0 && lanes == 0) return SPEC_OK;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState *d = nullptr;
    spec_status st = device_state(&d);
    if (st != SPEC_OK) return st;
    const int slots = (cols > 0 && k > 32) ? 2 : 1;
    const bool mapped = cols > 0 && id_map != nullptr;
    const int64_t max_ctas = (int64_t)d->sms * d->occ[slots - 1][mapped ? 1 : 0];
    const int64_t t_cols = lanes * (gamma + 1);

    RoundArgs a;
    memset(&a, 0, sizeof a);
    a.draft = draft; a.d_cols = cols; a.d_V = cols ? V : 1; a.k = cols ? k : 1;
    a.id_map = id_map; a.out_vals = vals; a.out_ids = ids;
    a.target = target; a.t_cols = t_cols; a.t_V = lanes ? tV : 1; a.gamma = gamma;
    a.drafts = drafts; a.out_accept = acc; a.out_commit = com;
    a.pstride = a.k + 2;
    split_warps(cols ? vectors_of(draft, cols * V) : 0, lanes ? vectors_of(target, t_cols * tV) : 0,
                max_ctas * kWarpsPerCta, a.pstride, INT64_MAX / 4, &a.d_warps, &a.t_warps);
    cudaStream_t stream = t_stream;
    const int64_t nwarps = (int64_t)a.d_warps + a.t_warps;
    const ScratchCaps need = {2 * (cols + t_cols), lanes, t_cols, nwarps * 2 * a.pstride};
    st = ensure_scratch(*d, need, stream);
    if (st != SPEC_OK) return st;
    const ScratchPtrs sp = scratch_ptrs(*d);
    a.partials = sp.partials;
    a.col_ticket = sp.col_ticket;
    a.col_cert = sp.col_ticket + (cols + t_cols);
    a.lane_ticket = sp.lane_ticket;
    a.t_argmax = sp.t_argmax;

    const dim3 grid((unsigned)((nwarps + kWarpsPerCta - 1) / kWarpsPerCta)), block(kThreads);
    if (slots == 1 && !mapped) spec_round_kernel<1, false><<<grid, block, kSmemBytes, stream>>>(a);
    else if (slots == 1) spec_round_kernel<1, true><<<grid, block, kSmemBytes, stream>>>(a);
    else if (!mapped) spec_round_kernel<2, false><<<grid, block, kSmemBytes, stream>>>(a);
    else spec_round_kernel<2, true><<<grid, block, kSmemBytes, stream>>>(a);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return SPEC_OK;
}

spec_status ensure_staging(DeviceState &d, size_t bytes)
{
    if (d.staging_bytes >= bytes) return SPEC_OK;
    cudaError_t e;
    if (d.staging) {
        e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
        cudaFree(d.staging);
        d.staging = nullptr;
        d.staging_bytes = 0;
    }
    e = cudaMalloc(&d.staging, bytes);
    if (e != cudaSuccess) {
        d.staging = nullptr;
        cudaGetLastError();
        return fail(SPEC_ERR_ALLOC, "cudaMalloc(%zu) for staging: %s", bytes, cudaGetErrorString(e));
    }
    d.staging_bytes = bytes;
    return SPEC_OK;
}

}  // namespace

// ---------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------

extern "C" {

spec_status spec_topk(const uint16_t *logits, int64_t cols, int64_t V, int32_t k, uint16_t *out_vals,
                      int32_t *out_ids)
{
    t_err.clear();
    spec_status st = check_topk_args(logits, cols, V, k, out_vals, out_ids);
    if (st != SPEC_OK) return st;
    return launch_round(logits, cols, V, k, nullptr, out_vals, out_ids, nullptr, nullptr, 0, 1, 1, nullptr,
                        nullptr);
}

spec_status spec_topk_mapped(const uint16_t *logits, int64_t cols, int64_t V, int32_t k, const int32_t *id_map,
                             uint16_t *out_vals, int32_t *out_ids)
{
    t_err.clear();
    spec_status st = check_topk_args(logits, cols, V, k, out_vals, out_ids);
    if (st != SPEC_OK) return st;
    if (cols > 0 && (!id_map || misaligned(id_map, 4))) return fail(SPEC_ERR_ARG, "id_map null or misaligned");
    return launch_round(logits, cols, V, k, cols > 0 ? id_map : nullptr, out_vals, out_ids, nullptr, nullptr, 0,
                        1, 1, nullptr, nullptr);
}

spec_status spec_verify_v(const uint16_t *target_logits, const int32_t *drafts, int64_t lanes, int32_t gamma,
                          int64_t V, int32_t *out_accept_len, int32_t *out_commit_ids)
{
    t_err.clear();
    spec_status st = check_verify_args(target_logits, drafts, lanes, gamma, V, out_accept_len, out_commit_ids);
    if (st != SPEC_OK) return st;
    return launch_round(nullptr, 0, 1, 1, nullptr, nullptr, nullptr, target_logits, drafts, lanes, gamma, V,
                        out_accept_len, out_commit_ids);
}

spec_status spec_verify(const uint16_t *target_logits, const int32_t *drafts, int64_t lanes, int32_t gamma,
                        int32_t *out_accept_len, int32_t *out_commit_ids)
{
    return spec_verify_v(target_logits, drafts, lanes, gamma, SPEC_VOCAB, out_accept_len, out_commit_ids);
}

spec_status spec_round(const uint16_t *draft_logits, int64_t cols, int64_t V, int32_t k, uint16_t *out_vals,
                       int32_t *out_ids, const uint16_t *target_logits, const int32_t *drafts, int64_t lanes,
                       int32_t gamma, int32_t *out_accept_len, int32_t *out_commit_ids)
{
    t_err.clear();
    spec_status st = check_topk_args(draft_logits, cols, V, k, out_vals, out_ids);
    if (st != SPEC_OK) return st;
    st = check_verify_args(target_logits, drafts, lanes, gamma, V, out_accept_len, out_commit_ids);
    if (st != SPEC_OK) return st;
    return launch_round(draft_logits, cols, V, k, nullptr, out_vals, out_ids, target_logits, drafts, lanes,
                        gamma, V, out_accept_len, out_commit_ids);
}

spec_status spec_round_host(const uint16_t *draft_logits, int64_t cols, int64_t V, int32_t k, uint16_t *out_vals,
                            int32_t *out_ids, const uint16_t *target_logits, const int32_t *drafts,
                            int64_t lanes, int32_t gamma, int32_t *out_accept_len, int32_t *out_commit_ids)
{
    t_err.clear();
    spec_status st = check_topk_args(draft_logits, cols, V, k, out_vals, out_ids);
    if (st != SPEC_OK) return st;
    st = check_verify_args(target_logits, drafts, lanes, gamma, V, out_accept_len, out_commit_ids);
    if (st != SPEC_OK) return st;
    if (cols == 0 && lanes == 0) return SPEC_OK;
    cudaStream_t stream = t_stream;
    if (stream_capturing(stream)) return fail(SPEC_ERR_ARG, "spec_round_host cannot be captured");
    const int64_t t_cols = lanes * (gamma + 1);
    const size_t b_dl = (size_t)cols * V * 2, b_tl = (size_t)t_cols * V * 2, b_dr = (size_t)lanes * gamma * 4;
    const size_t b_v = (size_t)cols * k * 2, b_i = (size_t)cols * k * 4, b_a = (size_t)lanes * 4,
                 b_c = (size_t)t_cols * 4;
    size_t off[7], tot = 0;
    const size_t sz[7] = {b_dl, b_tl, b_dr, b_v, b_i, b_a, b_c};
    for (int i = 0; i < 7; ++i) { off[i] = tot; tot = align256(tot + sz[i]); }
    char *s = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        DeviceState *d = nullptr;
        st = device_state(&d);
        if (st != SPEC_OK) return st;
        st = ensure_staging(*d, tot);
        if (st != SPEC_OK) return st;
        s = static_cast<char *>(d->staging);
    }
    cudaError_t e = cudaSuccess;
    if (cols) e = cudaMemcpyAsync(s + off[0], draft_logits, b_dl, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess && lanes) e = cudaMemcpyAsync(s + off[1], target_logits, b_tl, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess && lanes) e = cudaMemcpyAsync(s + off[2], drafts, b_dr, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync H2D");
    st = spec_round(cols ? (const uint16_t *)(s + off[0]) : nullptr, cols, V, k,
                    cols ? (uint16_t *)(s + off[3]) : nullptr, cols ? (int32_t *)(s + off[4]) : nullptr,
                    lanes ? (const uint16_t *)(s + off[1]) : nullptr, lanes ? (const int32_t *)(s + off[2]) : nullptr,
                    lanes, gamma, lanes ? (int32_t *)(s + off[5]) : nullptr, lanes ? (int32_t *)(s + off[6]) : nullptr);
    if (st != SPEC_OK) return st;
    if (cols) e = cudaMemcpyAsync(out_vals, s + off[3], b_v, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess && cols) e = cudaMemcpyAsync(out_ids, s + off[4], b_i, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess && lanes) e = cudaMemcpyAsync(out_accept_len, s + off[5], b_a, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess && lanes) e = cudaMemcpyAsync(out_commit_ids, s + off[6], b_c, cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync D2H");
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    return SPEC_OK;
}

spec_status spec_set_stream(void *stream)
{
    t_stream = static_cast<cudaStream_t>(stream);
    return SPEC_OK;
}

void *spec_get_stream(void) { return static_cast<void *>(t_stream); }

spec_status spec_reserve(int64_t max_cols, int32_t max_k, int64_t max_lanes, int32_t max_gamma)
{
    t_err.clear();
    if (max_cols < 0 || max_lanes < 0 || max_k < 1 || max_k > SPEC_MAX_K || max_gamma < 1 ||
        max_gamma > SPEC_MAX_GAMMA)
        return fail(SPEC_ERR_ARG, "spec_reserve: bad sizes");
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState *d = nullptr;
    spec_status st = device_state(&d);
    if (st != SPEC_OK) return st;
    const int64_t t_cols = max_lanes * (max_gamma + 1);
    const ScratchCaps need = {2 * (max_cols + t_cols), max_lanes, t_cols,
                              (int64_t)d->sms * d->occ[max_k > 32 ? 1 : 0][0] * kWarpsPerCta * 2 * (max_k + 2)};
    return ensure_scratch(*d, need, t_stream);
}

spec_status spec_release(void)
{
    t_err.clear();
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return SPEC_OK;
    DeviceState &d = g_dev[dev];
    if (!d.scratch && !d.staging) return SPEC_OK;
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    if (d.scratch) cudaFree(d.scratch);
    if (d.staging) cudaFree(d.staging);
    d.scratch = d.staging = nullptr;
    d.scratch_bytes = d.staging_bytes = 0;
    d.cap_cols = d.cap_lanes = d.cap_tcols = d.cap_part = 0;
    return SPEC_OK;
}

const char *spec_last_error(void) { return t_err.c_str(); }

int64_t spec_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

spec_status spec_device_status(void)
{
    t_err.clear();
    cudaError_t e = cudaStreamSynchronize(t_stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    unsigned int flags = 0, zero = 0;
    e = cudaMemcpyFromSymbol(&flags, g_wait_timeouts, sizeof flags);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyFromSymbol");
    if (flags == 0) return SPEC_OK;
    e = cudaMemcpyToSymbol(g_wait_timeouts, &zero, sizeof zero);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyToSymbol");
    return fail(SPEC_ERR_CUDA, "a kernel gave up a bounded wait on its copy pipeline; its results are invalid");
}

}  // extern "C"

// ---------------------------------------------------------------------------
// spec_round_noalloc: the same round, with its scratch in a fixed device array
// ---------------------------------------------------------------------------
//
// Some callers cannot let this library call cudaMalloc: an inference engine
// that hands out every byte of device memory from its own pool (a stray
// allocation breaks its accounting and can fail once the pool has taken the
// free memory), a serving loop that must never pay the device-wide
// synchronisation that cudaFree implies, or a C host that runs under a fixed
// memory budget.  For them this entry point keeps its scratch (column and lane
// tickets, target argmaxes, partial lists) in one statically sized device
// array, so it allocates nothing, ever.  The array costs every GPU that loads
// the library its size until the process exits.

namespace {

constexpr int64_t kNoAllocMaxCols = SPEC_NOALLOC_MAX_COLS;     // draft + target columns
constexpr int64_t kNoAllocMaxLanes = SPEC_NOALLOC_MAX_LANES;
constexpr int64_t kNoAllocPartials = 131072;                    // partial-list entries (1 MiB)
constexpr size_t kNoAllocColTicket = 0;
constexpr size_t kNoAllocLaneTicket = kNoAllocColTicket + ((2 * kNoAllocMaxCols * 4 + 255) & ~int64_t(255));
constexpr size_t kNoAllocArgmax = kNoAllocLaneTicket + ((kNoAllocMaxLanes * 4 + 255) & ~int64_t(255));
constexpr size_t kNoAllocPart = kNoAllocArgmax + ((kNoAllocMaxCols * 4 + 255) & ~int64_t(255));
constexpr size_t kNoAllocBytes = kNoAllocPart + kNoAllocPartials * 8;
constexpr size_t kNoAllocTicketBytes = kNoAllocArgmax;         // tickets and column certificates, cleared per call

// Device scratch of spec_round_noalloc.  In host code this name only stands
// for the symbol; the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

void *g_noalloc_ptr[kMaxDevices] = {};

// Once per device, with that device current: look up the array's address.
spec_status noalloc_scratch(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(SPEC_ERR_CUDA, "device ordinal %d unsupported", dev);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return SPEC_OK;
}

}  // namespace

extern "C" spec_status spec_round_noalloc(const uint16_t *draft_logits, int64_t cols, int64_t V, int32_t k,
                                          uint16_t *out_vals, int32_t *out_ids, const uint16_t *target_logits,
                                          const int32_t *drafts, int64_t lanes, int32_t gamma,
                                          int32_t *out_accept_len, int32_t *out_commit_ids)
{
    t_err.clear();
    spec_status st = check_topk_args(draft_logits, cols, V, k, out_vals, out_ids);
    if (st != SPEC_OK) return st;
    st = check_verify_args(target_logits, drafts, lanes, gamma, V, out_accept_len, out_commit_ids);
    if (st != SPEC_OK) return st;
    if (cols == 0 && lanes == 0) return SPEC_OK;
    const int64_t t_cols = lanes * (gamma + 1);
    if (cols + t_cols > kNoAllocMaxCols)
        return fail(SPEC_ERR_ARG, "spec_round_noalloc: %lld draft + target columns exceed its fixed scratch "
                    "limit of %lld", (long long)(cols + t_cols), (long long)kNoAllocMaxCols);
    if (lanes > kNoAllocMaxLanes)
        return fail(SPEC_ERR_ARG, "spec_round_noalloc: %lld lanes exceed its fixed scratch limit of %lld",
                    (long long)lanes, (long long)kNoAllocMaxLanes);

    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState *d = nullptr;
    st = device_state(&d);
    if (st != SPEC_OK) return st;
    void *base = nullptr;
    st = noalloc_scratch(&base);
    if (st != SPEC_OK) return st;

    const int slots = (cols > 0 && k > 32) ? 2 : 1;
    const int64_t max_ctas = (int64_t)d->sms * d->occ[slots - 1][0];
    RoundArgs a;
    memset(&a, 0, sizeof a);
    a.draft = draft_logits; a.d_cols = cols; a.d_V = cols ? V : 1; a.k = cols ? k : 1;
    a.out_vals = out_vals; a.out_ids = out_ids;
    a.target = target_logits; a.t_cols = t_cols; a.t_V = lanes ? V : 1; a.gamma = gamma;
    a.drafts = drafts; a.out_accept = out_accept_len; a.out_commit = out_commit_ids;
    a.pstride = a.k + 2;
    // warps as in spec_round, fewer if their published lists would not fit
    split_warps(cols ? vectors_of(draft_logits, cols * V) : 0, lanes ? vectors_of(target_logits, t_cols * V) : 0,
                max_ctas * kWarpsPerCta, a.pstride, kNoAllocPartials, &a.d_warps, &a.t_warps);
    const int64_t nwarps = (int64_t)a.d_warps + a.t_warps;
    char *p = static_cast<char *>(base);
    a.col_ticket = reinterpret_cast<unsigned int *>(p + kNoAllocColTicket);
    a.col_cert = a.col_ticket + (cols + t_cols);
    a.lane_ticket = reinterpret_cast<unsigned int *>(p + kNoAllocLaneTicket);
    a.t_argmax = reinterpret_cast<int32_t *>(p + kNoAllocArgmax);
    a.partials = reinterpret_cast<unsigned long long *>(p + kNoAllocPart);

    cudaStream_t stream = t_stream;
    // the array keeps whatever the last call left: start every ticket at zero
    cudaError_t e = cudaMemsetAsync(base, 0, kNoAllocTicketBytes, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(static scratch tickets)");
    const dim3 grid((unsigned)((nwarps + kWarpsPerCta - 1) / kWarpsPerCta)), block(kThreads);
    if (slots == 1) spec_round_kernel<1, false><<<grid, block, kSmemBytes, stream>>>(a);
    else spec_round_kernel<2, false><<<grid, block, kSmemBytes, stream>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return SPEC_OK;
}
