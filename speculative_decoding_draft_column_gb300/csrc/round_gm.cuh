// The group-maxima kernel: small rounds over vocabulary-sized columns, in one
// launch and two phases.
//
// Phase 1 streams.  The CTAs of a full-GPU grid each own a contiguous run of
// batches of the flat run of logits.  A batch is 512 * U 16-byte vectors;
// thread t of a CTA loads vectors t, t + 512, ..., t + 512 (U - 1) of it, one
// group of 8U elements, and keeps nothing but the group's maximum (one per
// column where the batch crosses a column boundary), written to global
// memory as a 2-byte order key.  The loads go out eight per thread at a time,
// then a bf16x2 max tree; there is no other work in the stream.
//
// Phase 2 selects, column by column, as soon as a column is complete: inside
// the stream for a column that lies in one CTA's slice, at the end of the
// slice for a column that CTAs share (a ticket per column: a CTA whose part
// of it ends inside its slice takes the ticket right there, the CTA whose
// part ends its slice comes last and finishes the column; a CTA that finds
// every other part in needs no atomic at all).  The finishing CTA loads the
// column's group keys, all at once, into shared memory.  Eight consecutive
// threads form a section; T, the kk-th largest of the 64 section maxima, is
// the key of kk distinct groups, so kk elements reach T and every one of the
// column's kk best elements lies in a group whose key reaches T: every group
// above T, and of the groups at T (ties) -- with token ids, which grow batch
// by batch -- those of the first batches that hold kk of them.  The CTA
// re-reads these groups from L2 with one 16-byte load per thread, collects
// their elements >= T and ranks them (value desc, id asc): ranks below kk
// are the column's top-kk in order.  Many candidates go through sorted lists
// per warp instead, merged at the end; more than the buffers hold, and the
// CTA scans the whole column exactly.  A target column then goes to greedy
// (or sampled) verify.  Every step of phase 2 issues its global loads
// together: a few round trips to L2 in all.  (That is slice mode; the
// kernel's other modes -- one pass, whole columns, finishing warps -- are
// described where they are defined, and the kernel's MODE parameter picks
// one.)
//
// The operations are those of the other two kernels ("A drafter inside the
// artifact", Ignis DFlash2 page, section "How it works"): top-k per draft
// column, largest first, ties to the smaller id; greedy verify.
#pragma once

#include "common.cuh"
#include "round_cta.cuh"

namespace gm {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kLoads = 8;             // 16-byte loads in flight per thread per step
constexpr int kCap = 4096;            // phase 2 candidate elements
constexpr int kGroupCap = 4096;       // phase 2 candidate groups
constexpr int kKeyRows = 64;          // batches of a column whose keys phase 2 keeps in shared memory
constexpr int kRankMax = 512;         // candidates ranked directly (more: sorted lists per warp)
constexpr int kFewTies = 64;          // groups at the bound all re-read up to this many
constexpr int64_t kMinV = 8 * 512;    // elements per column at least: a batch touches two columns at most

struct Smem {
    unsigned long long cand[kCap];
    unsigned long long wl[kWarps][SPEC_MAX_K];   // sorted lists, one per warp; wl[0] ends as the column's list
    uint32_t grp[kGroupCap];                     // candidate groups above the bound: (batch - first batch) << 9 | thread
    uint32_t tgrp[kGroupCap];                    // candidate groups at the bound (ties), the same way
    uint16_t keys[kKeyRows][512];                // the column's group keys, [batch - first batch][thread]
    uint32_t sec[64];                            // section maxima
    uint32_t smax[512];                          // the group-key maxima of the threads (or slots)
    uint32_t tiecnt[kKeyRows];                   // groups at the bound, per batch
    uint32_t wtie[kWarps];                       // groups at the bound, per warp
    int32_t wn[kWarps];
    uint32_t ncand, ngrp;                        // ngrp: groups above the bound (low 16 bits) and at it (high 16)
    uint32_t last[2];                            // the CTA completes its first / last column
};

constexpr size_t kSmemBytes = sizeof(Smem);
static_assert(kSmemBytes <= 227 * 1024, "one CTA per SM must fit");
static_assert(kKeyRows <= 64, "phase 2 marks a thread's batches in a 64-bit mask");

// One run (the draft or the target logits) on the 16-byte vector grid, as in
// the other kernels: vector j holds elements [8j - mis, 8j - mis + 8) of the
// flat run of N = cols * V elements; [jlo, jhi) lie wholly inside the buffer.
// Batches of 512 * U vectors, NB of them; CTA b owns batches
// [floor(b NB / W), floor((b + 1) NB / W)).
struct GmRun {
    const uint16_t *buf;
    const uint4 *vb;
    int64_t V, N, NV, jlo, jhi, NB;
    int64_t cols;            // N / V
    uint16_t *G;             // [NB][512]: group keys of each batch's first column
    uint16_t *H;             // [cols][512]: group keys of a column starting inside a batch, in that batch
    unsigned int *ticket;    // [cols]
    const int32_t *id_map;   // draft run only: local id -> vocabulary id (null: token ids)
    int W, kk, mis;
    bool draft;
};

__device__ __forceinline__ int64_t run_vectors(const uint16_t *buf, int64_t n)
{
    const int64_t mis = (int64_t)((reinterpret_cast<uintptr_t>(buf) >> 1) & 7);
    return n > 0 ? (n + mis + 7) >> 3 : 0;
}

template <int U>
__device__ __forceinline__ GmRun make_run(const RoundArgs &a, bool draft)
{
    constexpr int64_t B = 512 * U;
    const int64_t nbd = (run_vectors(a.draft, a.d_cols * a.d_V) + B - 1) / B;
    const int64_t nbt = (run_vectors(a.target, a.t_cols * a.t_V) + B - 1) / B;
    GmRun r;
    r.draft = draft;
    r.buf = draft ? a.draft : a.target;
    r.V = draft ? a.d_V : a.t_V;
    const int64_t cols = draft ? a.d_cols : a.t_cols;
    r.cols = cols;
    r.N = cols * r.V;
    r.W = draft ? a.d_units : a.t_units;
    r.kk = draft ? a.k : a.t_k;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(r.buf);
    r.mis = (int)((a0 >> 1) & 7);
    r.vb = reinterpret_cast<const uint4 *>(a0 - 2 * (uintptr_t)r.mis);
    r.NV = (r.N + r.mis + 7) >> 3;
    r.jlo = r.mis ? 1 : 0;
    r.jhi = ((r.N + r.mis) & 7) ? r.NV - 1 : r.NV;
    if (r.jhi < r.jlo) r.jhi = r.jlo;
    r.NB = draft ? nbd : nbt;
    uint16_t *hd = a.gkeys + (nbd + nbt) * 512;
    r.G = draft ? a.gkeys : a.gkeys + nbd * 512;
    r.H = draft ? hd : hd + a.d_cols * 512;
    r.ticket = a.col_ticket + (draft ? 0 : a.d_cols);
    r.id_map = draft ? a.id_map : nullptr;
    return r;
}

// elements [elem_lo, elem_hi) of batch g; the batch holding element e
template <int U>
__device__ __forceinline__ int64_t elem_lo(const GmRun &r, int64_t g)
{
    const int64_t e = 8 * g * (512 * U) - r.mis;
    return e > 0 ? e : 0;
}
template <int U>
__device__ __forceinline__ int64_t elem_hi(const GmRun &r, int64_t g)
{
    const int64_t e = 8 * (g + 1) * (512 * U) - r.mis;
    return e < r.N ? e : r.N;
}
template <int U>
__device__ __forceinline__ int64_t batch_of(const GmRun &r, int64_t e) { return ((e + r.mis) >> 3) / (512 * U); }

__device__ __forceinline__ int64_t slice_lo(const GmRun &r, int64_t b) { return udiv(b * r.NB, r.W); }
__device__ __forceinline__ int64_t owner_of(const GmRun &r, int64_t g) { return udiv((g + 1) * r.W - 1, r.NB); }

__device__ __forceinline__ uint32_t key_of(uint32_t m2) { return order_key(hmax_splat(m2) & 0xFFFFu); }

// Fold vector q (elements [g0, g0 + 8)) into the maxima of the column
// before element cut (ma) and of the one from it on (mb).
__device__ __forceinline__ void split_max(const uint4 &q, int64_t g0, int64_t cut, uint32_t &ma, uint32_t &mb)
{
    if (g0 + 8 <= cut) {
        ma = bmax2(ma, vmax(q));
    } else if (g0 >= cut) {
        mb = bmax2(mb, vmax(q));
    } else {
        const int s = (int)(cut - g0);   // elements [0, s) before the cut
        const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
        uint32_t wa[4], wb[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const bool lo_a = 2 * h < s, hi_a = 2 * h + 1 < s;
            wa[h] = (lo_a ? (wd[h] & 0xFFFFu) : 0x7FFFu) | (hi_a ? (wd[h] & 0xFFFF0000u) : 0x7FFF0000u);
            wb[h] = (lo_a ? 0x7FFFu : (wd[h] & 0xFFFFu)) | (hi_a ? 0x7FFF0000u : (wd[h] & 0xFFFF0000u));
        }
        ma = bmax2(ma, bmax2(bmax2(wa[0], wa[1]), bmax2(wa[2], wa[3])));
        mb = bmax2(mb, bmax2(bmax2(wb[0], wb[1]), bmax2(wb[2], wb[3])));
    }
}

// Phase 1, one step: the kLoads vectors of every thread in batches
// [gb, gb + 8 / U) of the slice (which ends at batch g1b); each group's key
// to G, and to H where a batch crosses into the next column.  cn is the
// column after the one in progress and cut its first element.
template <int U>
__device__ __forceinline__ void stream_step(const GmRun &r, int64_t gb, int64_t g1b, int64_t &cn, int64_t &cut)
{
    constexpr int P = kLoads / U;
    constexpr int64_t B = 512 * U;
    const int t = threadIdx.x;
    uint4 q[kLoads];
#pragma unroll
    for (int v = 0; v < kLoads; ++v) {
        const int64_t j = (gb + v / U) * B + (v % U) * 512 + t;
        q[v] = (gb + v / U < g1b && j >= r.jlo && j < r.jhi) ? __ldg(r.vb + j) : make_uint4(kNaN2, kNaN2, kNaN2, kNaN2);
    }
    if (gb * B < r.jlo || (gb + P) * B > r.jhi) {
        // the buffer's edge vectors (at most one at each end), element by element
#pragma unroll
        for (int v = 0; v < kLoads; ++v) {
            const int64_t j = (gb + v / U) * B + (v % U) * 512 + t;
            if (gb + v / U < g1b && j < r.NV && (j < r.jlo || j >= r.jhi)) q[v] = load_edge(r.buf, j, r.mis, 0, r.N);
        }
    }
#pragma unroll
    for (int p = 0; p < P; ++p) {
        const int64_t g = gb + p;
        if (g >= g1b) break;
        const int64_t e1 = elem_hi<U>(r, g);
        uint32_t ma = kNaN2, mb = kNaN2;
        if (e1 <= cut) {
#pragma unroll
            for (int u = 0; u < U; ++u) ma = bmax2(ma, vmax(q[p * U + u]));
        } else {
#pragma unroll
            for (int u = 0; u < U; ++u) split_max(q[p * U + u], 8 * (g * B + u * 512 + t) - r.mis, cut, ma, mb);
            r.H[cn * 512 + t] = (uint16_t)key_of(mb);
        }
        r.G[g * 512 + t] = (uint16_t)key_of(ma);
        if (e1 >= cut) {   // the next batch starts in column cn
            ++cn;
            cut += r.V;
        }
    }
}

// The largest T such that at least kk of the 64 values {v0, v1 of every
// lane} reach T (the kk-th largest; 1 <= kk <= 64): a bisection between the
// smallest and the largest value, in every lane of the warp (the values
// cluster: a few steps).
__device__ __forceinline__ uint32_t kth_of_64(uint32_t v0, uint32_t v1, int kk)
{
    uint32_t lo = __reduce_min_sync(kFull, v0 < v1 ? v0 : v1);   // all 64 reach it
    uint32_t hi = __reduce_max_sync(kFull, v0 > v1 ? v0 : v1);
    if (kk == 1) return hi;
    while (lo < hi) {
        const uint32_t mid = (lo + hi + 1) >> 1;
        const int n = __popc(__ballot_sync(kFull, v0 >= mid)) + __popc(__ballot_sync(kFull, v1 >= mid));
        if (n >= kk) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// Append the groups of this thread's rows in above and tie (bit i: batch i
// of the column) to the two group lists, one shared atomic per warp on the
// packed count (above: low 16 bits, ties: high 16 bits; at most 512 * 64 of
// each).
__device__ __forceinline__ void append_groups(Smem &s, unsigned long long above, unsigned long long tie, int lane)
{
    int total;
    const int excl = warp_exclusive_sum(__popcll(above) | (__popcll(tie) << 16), lane, total);
    if (total == 0) return;
    uint32_t base = 0;
    if (lane == 0) base = atomicAdd(&s.ngrp, (uint32_t)total);
    base = __shfl_sync(kFull, base, 0) + (uint32_t)excl;
    uint32_t pa = base & 0xFFFFu, pt = base >> 16;
    const uint32_t tid = threadIdx.x & 511u;
    for (unsigned long long m = above; m; m &= m - 1, ++pa)
        if (pa < (uint32_t)kGroupCap) s.grp[pa] = ((uint32_t)(__ffsll((long long)m) - 1) << 9) | tid;
    for (unsigned long long m = tie; m; m &= m - 1, ++pt)
        if (pt < (uint32_t)kGroupCap) s.tgrp[pt] = ((uint32_t)(__ffsll((long long)m) - 1) << 9) | tid;
}

// The kk-th largest of the n values v[0 .. n) (n a multiple of 32, at most
// 512), in every lane of the warp: a bisection between the smallest and the
// largest.  For kk above 8, where 64 section maxima bound too loosely.
__device__ __forceinline__ uint32_t kth_of_smem(const uint32_t *v, int n, int kk, int lane)
{
    uint32_t x[16];
    uint32_t lo = 0xFFFFFFFFu, hi = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        x[i] = i * 32 < n ? v[i * 32 + lane] : 0u;
        if (i * 32 < n) {
            lo = x[i] < lo ? x[i] : lo;
            hi = x[i] > hi ? x[i] : hi;
        }
    }
    lo = __reduce_min_sync(kFull, lo);   // all n values reach it
    hi = __reduce_max_sync(kFull, hi);
    while (lo < hi) {
        const uint32_t mid = (lo + hi + 1) >> 1;
        uint32_t cnt = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) cnt += (i * 32 < n && x[i] >= mid) ? 1u : 0u;
        if ((int)__reduce_add_sync(kFull, cnt) >= kk) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// Append group id gid of this lane (if take) to the group list, one shared
// atomic per warp.
__device__ __forceinline__ void append_group(Smem &s, bool take, uint32_t gid, int lane)
{
    const uint32_t bal = __ballot_sync(kFull, take);
    if (!bal) return;
    uint32_t base = 0;
    if (lane == 0) base = atomicAdd(&s.ngrp, (uint32_t)__popc(bal));
    base = __shfl_sync(kFull, base, 0);
    const uint32_t pos = base + (uint32_t)__popc(bal & lanemask_lt());
    if (take && pos < (uint32_t)kGroupCap) s.grp[pos] = gid;
}

// What phase 2's rare paths need of a run, passed by value (a GmRun passed
// by reference would have to live in local memory).
struct RunView {
    const uint16_t *buf;
    const uint4 *vb;
    const int32_t *id_map;
    int64_t jlo, jhi;
    int mis, kk;
};

__device__ __forceinline__ RunView view_of(const GmRun &r)
{
    return RunView{r.buf, r.vb, r.id_map, r.jlo, r.jhi, r.mis, r.kk};
}

// Vector j restricted to column [cb, ce): elements outside it (or outside
// the buffer) as NaN.
__device__ __forceinline__ uint4 load_col_vec(const RunView &v, int64_t j, int64_t cb, int64_t ce)
{
    const int64_t g0 = 8 * j - v.mis;
    if (j >= v.jlo && j < v.jhi && g0 >= cb && g0 + 8 <= ce) return __ldg(v.vb + j);
    return load_edge(v.buf, j, v.mis, cb, ce);
}

__device__ __forceinline__ uint32_t half_of(const uint4 &q, int e)
{
    const uint32_t w = (e & 4) ? ((e & 2) ? q.w : q.z) : ((e & 2) ? q.y : q.x);
    return (e & 1) ? (w >> 16) : (w & 0xFFFFu);
}

// Vector u of a thread's registers, u not known at compile time (selects:
// a short, branch-free sequence instead of a copy of the caller's code per
// vector).
template <int L>
__device__ __forceinline__ uint4 pick(const uint4 (&q)[L], int u)
{
    uint4 v = q[0];
#pragma unroll
    for (int i = 1; i < L; ++i)
        if (i == u) v = q[i];
    return v;
}

__device__ __forceinline__ unsigned long long make_entry(uint32_t key, uint32_t id, uint32_t raw)
{
    return ((unsigned long long)key << 48) | ((unsigned long long)(~id) << 16) | raw;
}

// Rank each of the n candidates in s.cand (n <= kRankMax, all distinct)
// among them, value desc, id asc, and put those ranked below kk into
// s.wl[0] in order.  Thread t of a team of nt threads; the candidates are
// compared four at a time (two 16-byte shared loads, four independent
// counts).
__device__ __forceinline__ void rank_into_list(Smem &s, int n, int kk, int t, int nt)
{
    const ulonglong2 *c2 = reinterpret_cast<const ulonglong2 *>(s.cand);
    for (int i = t; i < n; i += nt) {
        const unsigned long long e = s.cand[i];
        int r0 = 0, r1 = 0, r2 = 0, r3 = 0;
        int j = 0;
        for (; j + 4 <= n; j += 4) {
            const ulonglong2 a = c2[j >> 1], b = c2[(j >> 1) + 1];
            r0 += a.x > e ? 1 : 0;
            r1 += a.y > e ? 1 : 0;
            r2 += b.x > e ? 1 : 0;
            r3 += b.y > e ? 1 : 0;
        }
        for (; j < n; ++j) r0 += s.cand[j] > e ? 1 : 0;
        const int rank = r0 + r1 + r2 + r3;
        if (rank < kk) s.wl[0][rank] = e;
    }
}

// A barrier of a team of NW warps: the CTA (id 0) or a named barrier.
template <int NW, int BAR>
__device__ __forceinline__ void team_sync()
{
    if constexpr (BAR == 0) __syncthreads();
    else asm volatile("bar.sync %0, %1;" ::"n"(BAR), "n"(NW * 32) : "memory");
}

// Warp 0 of a team of NW warps merges the team's sorted lists (s.wl[w][0 ..
// s.wn[w]), w the warp within the team) into s.wl[0]: the kk best of all of
// them.  Every thread of the team must call it.
template <int NW, int BAR>
__device__ __forceinline__ void merge_lists(Smem &s, int kk, int lane, int w)
{
    team_sync<NW, BAR>();
    if (w != 0) return;
    int n0 = s.wn[0];
    for (int q = 1; q < NW; ++q) {
        const int nq = s.wn[q];
        for (int b2 = 0; b2 < nq; b2 += 32) {
            unsigned long long e = b2 + lane < nq ? s.wl[q][b2 + lane] : 0ull;
            if (n0 == kk && e < s.wl[0][kk - 1]) e = 0ull;
            n0 = cta::list_merge32(s.wl[0], n0, e, kk, lane);
        }
    }
}

// The kk best of the n candidates in s.cand (many of them: ties at the
// bound), into s.wl[0]: every warp of the team folds a share into its own
// sorted list, behind the list's kk-th entry, then the lists are merged.
template <int NW, int BAR>
__device__ __noinline__ void select_many(int n, int kk, Smem &s, int lane, int w)
{
    unsigned long long *wl = s.wl[w];
    int nw = 0;
    for (int base = 32 * w; base < n; base += NW * 32) {
        unsigned long long e = base + lane < n ? s.cand[base + lane] : 0ull;
        if (nw == kk && e < wl[kk - 1]) e = 0ull;
        nw = cta::list_merge32(wl, nw, e, kk, lane);
    }
    if (lane == 0) s.wn[w] = nw;
    merge_lists<NW, BAR>(s, kk, lane, w);
}

// Exact top-kk of the elements [cb, ce) of a column (its ids counted from
// element idb) among those >= T, for any input (the path for massive ties):
// every warp scans a share of the range's vectors into its own sorted list,
// keeping only entries above the list's kk-th; the lists are then merged
// into s.wl[0].  Every thread of the team (NW warps) must call it.
template <int NW, int BAR>
__device__ __noinline__ void exact_scan(const RunView r, int64_t cb, int64_t ce, int64_t idb, uint32_t T, Smem &s,
                                        int lane, int w)
{
    const int kk = r.kk;
    unsigned long long *wl = s.wl[w];
    int nw = 0;
    unsigned long long thr = 0ull;   // a full list's kk-th entry: only better entries can enter
    const int64_t jf = (cb + r.mis) >> 3, jl = (ce - 1 + r.mis) >> 3;
    for (int64_t base = jf + 32 * w; base <= jl; base += NW * 32) {
        const int64_t j = base + lane;
        const uint4 q = j <= jl ? load_col_vec(r, j, cb, ce) : make_uint4(kNaN2, kNaN2, kNaN2, kNaN2);
        const int64_t g0 = 8 * j - r.mis;
#pragma unroll 1
        for (int e = 0; e < 8; ++e) {
            const uint32_t raw = half_of(q, e);
            const uint32_t key = order_key(raw);
            unsigned long long cand = 0ull;
            if (key != 0 && key >= T && key >= entry_key(thr)) {
                uint32_t id = (uint32_t)(g0 + e - idb);
                if (r.id_map) id = (uint32_t)__ldg(r.id_map + id);
                cand = make_entry(key, id, raw);
                if (cand < thr) cand = 0ull;
            }
            if (__ballot_sync(kFull, cand != 0ull)) {
                nw = cta::list_merge32(wl, nw, cand, kk, lane);
                thr = nw == kk ? wl[kk - 1] : 0ull;
            }
        }
    }
    if (lane == 0) s.wn[w] = nw;
    merge_lists<NW, BAR>(s, kk, lane, w);
}

__device__ __forceinline__ uint32_t ld_relaxed_u32(const unsigned int *p)
{
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Target column c (position j of lane ln) is decided: its commit token and
// whether draft j was accepted (greedy verify: the argmax and whether it
// equals draft j; sampled verify: see sampled_decide).  Warp-wide.  No fence
// anywhere: the column leaves token + 2 (never 0) in its slot of the lane
// (the column-certificate words, zero between launches), then adds to the
// lane's ticket word, relaxed: 1 (bits 0-7: positions done) and bit 8 + j
// if accepted.  The last position's warp computes the accept length acc
// from the word, reads every slot of the lane -- waiting (bounded) for one
// that is not visible yet, since its column took the ticket after writing
// it -- clears them, and writes all commit ids: each position's token up to
// acc (below acc the accepted drafts), -1 after it.  A column's own commit
// id is thus only ever written by the lane's last position.
__device__ __forceinline__ void lane_done(const RoundArgs &a, int64_t c, int32_t token, bool accepted, int lane)
{
    const int gamma = a.gamma, gp1 = gamma + 1;
    const int64_t ln = udiv(c, gp1);
    const int j = (int)(c - ln * gp1);
    unsigned int *slot = a.col_cert + a.d_cols + ln * gp1;
    uint32_t word = 0;
    if (lane == 0) {
        asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(slot + j), "r"((uint32_t)token + 2u) : "memory");
        const uint32_t add = 1u + ((accepted ? 1u : 0u) << (8 + j));
        asm volatile("atom.relaxed.gpu.global.add.u32 %0, [%1], %2;" : "=r"(word) : "l"(a.lane_ticket + ln), "r"(add)
                     : "memory");
        word += add;
    }
    word = __shfl_sync(kFull, word, 0);
    if ((word & 0xFFu) != (uint32_t)gp1) return;
    const uint32_t flags = (word >> 8) & ((1u << gamma) - 1u);
    const int acc = __ffs(~flags) - 1 < gamma ? __ffs(~flags) - 1 : gamma;
    if (lane < gp1) {
        uint32_t v = ld_relaxed_u32(slot + lane);
        if (v == 0u) {
            const uint64_t t0 = global_ns();
            while ((v = ld_relaxed_u32(slot + lane)) == 0u) {
                if (global_ns() - t0 > kWaitLimitNs) {
                    atomicOr(&g_wait_timeouts, 1u);
                    v = 1u;   // commit id -1
                    break;
                }
            }
        }
        slot[lane] = 0u;   // after the read of the column's value: ready for the next launch
        a.out_commit[ln * gp1 + lane] = lane <= acc ? (int32_t)(v - 2u) : -1;
    }
    count_lane(a.counters, gamma, acc, lane);
    if (lane == 0) {
        a.out_accept[ln] = acc;
        a.lane_ticket[ln] = 0u;   // ready for the next launch
    }
}

// What the candidate steps of phase 2 leave for the last one.
struct Sel {
    uint32_t T;          // the bound
    int upto;            // groups at T taken from batches below upto only
    bool lost;           // a list overflowed: scan the column instead
    int32_t draft_tok;   // (thread 0) a target column's draft token; -2: none
};

// Phase 2 up to the candidates of column c (every thread of the CTA calls
// it), over the column's first `rows` batches: the bound, the groups that
// can hold a winner, and their elements >= T in the candidate buffer.  The
// caller adds the candidates of later batches, if any, and calls rank_emit.
template <int U, bool COLS>
__device__ __forceinline__ Sel select_candidates(const RoundArgs &a, const GmRun &r, int64_t c, int rows, Smem &s,
                                                 int first = 0)
{
    constexpr int64_t B = 512 * U;
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const int kk = r.kk;
    const int64_t cb = c * r.V, ce = cb + r.V;
    // the column's groups: batch i (of nb), thread t' = vectors jbase + i B + u 512 + t'
    int64_t jbase;
    int nb;
    const uint16_t *k0 = nullptr, *kr = nullptr;   // slice mode: keys of batch 0, and of batch i at kr[512 i]
    if (COLS) {   // (from batch `first` of the column on: a part of it, in the cluster modes)
        jbase = (cb + r.mis) >> 3;
        nb = (int)((((ce - 1 + r.mis) >> 3) - jbase) / B + 1) - first;
        jbase += (int64_t)first * B;
    } else {
        const int64_t bf = batch_of<U>(r, cb), bl = batch_of<U>(r, ce - 1);
        const bool hin = elem_lo<U>(r, bf) < cb;   // the column starts inside batch bf: its keys there are in H
        jbase = bf * B;
        nb = (int)(bl - bf + 1);
        k0 = hin ? r.H + c * 512 + t : r.G + bf * 512 + t;
        kr = r.G + bf * 512 + t;
    }
    if (nb > rows) nb = rows;
    const RunView rv = view_of(r);
    // a target column's draft token (-2: none, the bonus position), early
    int32_t draft_tok = -2;
    if (!r.draft && t == 0) {
        const int gp1 = a.gamma + 1;
        const int64_t ln = udiv(c, gp1);
        const int j = (int)(c - ln * gp1);
        if (j < a.gamma) draft_tok = __ldg(a.drafts + ln * a.gamma + j);
    }
    __syncthreads();
    if (t < kKeyRows) s.tiecnt[t] = 0u;

    // 1. the column's group keys in shared memory (the first kKeyRows
    //    batches; column mode: there already, from the stream; slice mode:
    //    sixteen loads in flight per thread); this thread's maximum
    uint32_t mt = 0;
    if (COLS) {
        for (int i = 0; i < nb; ++i) {
            const uint32_t key = s.keys[i][t];
            mt = key > mt ? key : mt;
        }
    } else {
        for (int i0 = 0; i0 < nb; i0 += 16) {
            uint32_t kv[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) kv[q] = i0 + q < nb ? __ldcg(i0 + q == 0 ? k0 : kr + 512 * (i0 + q)) : 0u;
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                mt = kv[q] > mt ? kv[q] : mt;
                if (i0 + q < kKeyRows) s.keys[i0 + q][t] = (uint16_t)kv[q];
            }
        }
    }
    // 2. the bound T: the kk-th largest section maximum (sections of 8 threads)
    uint32_t m8 = mt;
#pragma unroll
    for (int d = 1; d < 8; d <<= 1) {
        const uint32_t o = __shfl_xor_sync(kFull, m8, d);
        m8 = o > m8 ? o : m8;
    }
    if ((lane & 7) == 0) s.sec[4 * w + (lane >> 3)] = m8;
    s.smax[t] = mt;
    if (t == 0) s.cand[0] = ~0ull;   // kk = 1: the shared minimum below
    __syncthreads();
    // T: the kk-th largest of 64 section maxima (kk <= 8) or of the 512
    // threads' maxima; either is the key of kk distinct groups
    const uint32_t T = kk <= 8 ? kth_of_64(s.sec[lane], s.sec[lane + 32], kk) : kth_of_smem(s.smax, kThreads, kk, lane);
    if (kk == 1 && r.id_map == nullptr && nb <= kKeyRows) {
        // the column's maximum T (an argmax: greedy verify, or a top-1):
        // each thread with a group at T reads its first such group again
        // (its groups are in position order) and offers the first element
        // at T in it; a shared minimum of (position, value) picks the
        // smallest id.  One candidate, no group list, no rank.
        if (mt != 0 && mt == T) {
            int i = 0;
            while (i < nb - 1 && s.keys[i][t] != T) ++i;
            const int64_t jg = jbase + (int64_t)i * B + t;
            uint4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) v[u] = load_col_vec(rv, jg + u * 512, cb, ce);
            uint32_t um = 0;
#pragma unroll
            for (int u = 0; u < U; ++u) um |= key_of(vmax(v[u])) == T ? 1u << u : 0u;
            const int u = __ffs(um) - 1;
            const uint4 x = pick(v, u);
            int e = 7;
#pragma unroll 1
            for (int k2 = 6; k2 >= 0; --k2)
                if (order_key(half_of(x, k2)) == T) e = k2;
            const int64_t pos = 8 * (jg + u * 512) - r.mis + e - cb;
            atomicMin(&s.cand[0], ((unsigned long long)pos << 16) | half_of(x, e));
        }
        __syncthreads();
        if (t == 0) {
            const unsigned long long b = s.cand[0];
            s.cand[0] = make_entry(T, (uint32_t)(b >> 16), (uint32_t)(b & 0xFFFFu));
            s.ncand = b != ~0ull ? 1u : 0u;
        }
        return Sel{T, 1 << 30, false, draft_tok};
    }
    // 3. the groups to re-read: every group above T, and of the groups at T
    //    (ties) -- with token ids, which grow batch by batch, and more than a
    //    few of them -- only those of the first batches that hold kk of them
    //    (they hold kk elements at T, all with smaller ids than any tie
    //    further on).  Each thread marks its rows above / at T in two masks;
    //    one shared atomic per warp appends a mask's groups.
    int upto = 1 << 30;   // groups at T taken from batches below upto only
    if (nb > kKeyRows) {
        // a column of more than kKeyRows batches: every group reaching T, in
        // the first list (a plain count)
        if (__ballot_sync(kFull, mt != 0 && mt >= T) != 0u)
#pragma unroll 1
            for (int i = 0; i < nb; ++i) {
                const uint32_t key = i < kKeyRows ? s.keys[i][t] : __ldcg(i == 0 ? k0 : kr + 512 * i);
                append_group(s, key != 0 && key >= T, ((uint32_t)i << 9) | (uint32_t)t, lane);
            }
        __syncthreads();
    } else {
        unsigned long long above = 0ull, tie = 0ull;
        if (mt != 0 && mt >= T)
#pragma unroll 1
            for (int i = 0; i < nb; ++i) {
                const uint32_t key = s.keys[i][t];
                above |= (unsigned long long)(key != 0 && key > T) << i;
                tie |= (unsigned long long)(key != 0 && key == T) << i;
            }
        append_groups(s, above, tie, lane);
        __syncthreads();
        if (r.id_map == nullptr && (s.ngrp >> 16) > (uint32_t)kFewTies) {
            // many ties: groups at T per batch, then the list of groups at T
            // again, from the first batches holding kk of them only
#pragma unroll 1
            for (int i = 0; i < nb; ++i) {
                const uint32_t ni = (uint32_t)__popc(__ballot_sync(kFull, (tie >> i) & 1ull));
                if (lane == 0 && ni) atomicAdd(&s.tiecnt[i], ni);
            }
            __syncthreads();
            int acc = 0;
            for (int i = 0; i < nb; ++i) {
                acc += (int)s.tiecnt[i];
                if (acc >= kk) {
                    upto = i + 1;
                    break;
                }
            }
            const uint32_t keep_above = s.ngrp & 0xFFFFu;
            __syncthreads();   // every thread has read the count
            if (t == 0) s.ngrp = keep_above;
            __syncthreads();
            append_groups(s, 0ull, upto >= 64 ? tie : tie & ((1ull << upto) - 1ull), lane);
            __syncthreads();
        }
    }
    const int na = nb > kKeyRows ? (int)s.ngrp : (int)(s.ngrp & 0xFFFFu);
    const int nt = nb > kKeyRows ? 0 : (int)(s.ngrp >> 16);
    const int ng = na + nt;
    // 4. their elements >= T: one 16-byte vector per thread per pass, up to
    //    four passes' loads in flight
    if (na <= kGroupCap && nt <= kGroupCap) {
        const int nv = ng * U;
        for (int p0 = 0; p0 < nv; p0 += 4 * kThreads) {
            uint4 q[4];
            int64_t jv[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const int p = p0 + h * kThreads + t;
                jv[h] = -1;
                q[h] = make_uint4(kNaN2, kNaN2, kNaN2, kNaN2);
                const bool at_t = p / U >= na;   // a group at T: only from the batches below upto
                const uint32_t gid = p < nv ? (at_t ? s.tgrp[p / U - na] : s.grp[p / U]) : 0u;
                if (p < nv && (!at_t || (int)(gid >> 9) < upto)) {
                    const int64_t j = jbase + (int64_t)(gid >> 9) * B + (p % U) * 512 + (gid & 511u);
                    if (j < r.NV) {
                        jv[h] = j;
                        q[h] = load_col_vec(rv, j, cb, ce);
                    }
                }
            }
#pragma unroll 1
            for (int h = 0; h < 4; ++h) {
                if (p0 + h * kThreads + 32 * w >= nv) break;   // this warp has no vector in the pass
                const uint4 qh = h == 0 ? q[0] : h == 1 ? q[1] : h == 2 ? q[2] : q[3];
                const int64_t g0 = 8 * (h == 0 ? jv[0] : h == 1 ? jv[1] : h == 2 ? jv[2] : jv[3]) - r.mis;
                uint32_t mask = 0;   // this lane's elements >= T
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const uint32_t key = order_key(half_of(qh, e));
                    mask |= (key != 0 && key >= T) ? 1u << e : 0u;
                }
                int total;
                const int excl = warp_exclusive_sum(__popc(mask), lane, total);
                if (total == 0) continue;
                uint32_t pos = 0;
                if (lane == 0) pos = atomicAdd(&s.ncand, (uint32_t)total);
                pos = __shfl_sync(kFull, pos, 0) + (uint32_t)excl;
                for (uint32_t m = mask; m; m &= m - 1, ++pos) {
                    const int e = __ffs(m) - 1;
                    const uint32_t raw = half_of(qh, e);
                    uint32_t id = (uint32_t)(g0 + e - cb);
                    if (r.id_map) id = (uint32_t)__ldg(r.id_map + id);
                    if (pos < (uint32_t)kCap) s.cand[pos] = make_entry(order_key(raw), id, raw);
                }
            }
        }
    }
    return Sel{T, upto, na > kGroupCap || nt > kGroupCap, draft_tok};
}

// Phase 2, the last step for column c: the kk best of the candidates, in
// order, to the outputs (draft) or to verify (target); the column's ticket
// cleared if shared.  Every thread of the CTA calls it.
template <int U>
__device__ __forceinline__ void rank_emit(const RoundArgs &a, const GmRun &r, int64_t c, bool shared, const Sel &sel,
                                          Smem &s)
{
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const int kk = r.kk;
    const int64_t cb = c * r.V, ce = cb + r.V;
    const uint32_t T = sel.T;
    const int32_t draft_tok = sel.draft_tok;
    const RunView rv = view_of(r);
    __syncthreads();
    const int n = (int)s.ncand;
    if (sel.lost || n > kCap) {
        exact_scan<kWarps, 0>(rv, cb, ce, cb, T, s, lane, w);
    } else if (n > kRankMax) {
        select_many<kWarps, 0>(n, kk, s, lane, w);
    } else {
        rank_into_list(s, n, kk, t, kThreads);
    }
    __syncthreads();
    if (r.draft) {
        for (int i = t; i < kk; i += kThreads) {
            const unsigned long long e = s.wl[0][i];
            a.out_vals[c * kk + i] = entry_raw(e);
            a.out_ids[c * kk + i] = (int32_t)entry_id(e);
        }
    } else if (w == 0) {
        int32_t token = (int32_t)entry_id(s.wl[0][0]);
        bool accepted;
        if (a.uniforms) accepted = sampled_decide(a, c, s.wl[0], kk, lane, token);
        else accepted = __shfl_sync(kFull, draft_tok, 0) == token;
        lane_done(a, c, token, accepted, lane);
    }
    if (t == 0) {
        s.ncand = 0u;
        s.ngrp = 0u;
        if (shared) r.ticket[c] = 0u;   // ready for the next launch
    }
    __syncthreads();
}

// Phase 2 for column c of run r, all of it (every thread of the CTA calls
// it).  shared: the column's ticket is to be cleared for the next launch.
// Every key of the column is written (this CTA's own keys: before the
// barrier at entry).
template <int U, bool COLS>
__device__ __forceinline__ void finish_column(const RoundArgs &a, const GmRun &r, int64_t c, bool shared, Smem &s)
{
    const Sel sel = select_candidates<U, COLS>(a, r, c, 1 << 30, s);
    rank_emit<U>(a, r, c, shared, sel, s);
}

// Column c's CTAs: those owning its first and last batch.
template <int U>
__device__ __forceinline__ void column_owners(const GmRun &r, int64_t c, int64_t &wf, int64_t &wl)
{
    wf = owner_of(r, batch_of<U>(r, c * r.V));
    wl = owner_of(r, batch_of<U>(r, (c + 1) * r.V - 1));
}

__device__ __forceinline__ uint32_t ld_acquire(const unsigned int *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Thread 0, at the end of the slice, for a shared column whose part here is
// written (others = the number of other CTAs that share it): true if this
// CTA is to finish the column.  If every other part is in already, it is,
// with no atomic (its own keys need no release: only it reads them);
// otherwise it takes the ticket, and finishes if it comes last.
__device__ __forceinline__ uint32_t arrive_at_end(unsigned int *ticket, uint32_t others)
{
    if (ld_acquire(ticket) == others) return 1u;
    return atom_add_acq_rel(ticket, 1u) == others ? 1u : 0u;
}

// Column mode (U = 8): CTA b owns whole columns [floor(b cols / W),
// floor((b + 1) cols / W)) of its run and streams them one by one in
// batches counted from each column's first vector, writing the group keys
// straight into shared memory; every column is finished right after its
// last batch, by the CTA alone (no tickets, no keys in global memory).
template <int U>
__device__ __forceinline__ void stream_columns(const RoundArgs &a, const GmRun &r, int bi, Smem &s)
{
    constexpr int P = kLoads / U;
    constexpr int64_t B = 512 * U;
    static_assert(P == 1, "column mode: one batch per step");
    const int t = threadIdx.x;
    const int64_t cols = r.cols;
    const int64_t c0 = udiv(bi * cols, r.W), c1 = udiv((bi + 1) * cols, r.W);
    for (int64_t c = c0; c < c1; ++c) {
        const int64_t cb = c * r.V, ce = cb + r.V;
        const int64_t jf = (cb + r.mis) >> 3, jl = (ce - 1 + r.mis) >> 3;
        const int nb = (int)((jl - jf) / B + 1);
        for (int i0 = 0; i0 < nb; i0 += P) {
            uint4 q[kLoads];
#pragma unroll
            for (int v = 0; v < kLoads; ++v) {
                const int64_t j = jf + (int64_t)(i0 + v / U) * B + (v % U) * 512 + t;
                q[v] = (i0 + v / U < nb && j > jf && j < jl && j >= r.jlo && j < r.jhi)
                           ? __ldg(r.vb + j) : make_uint4(kNaN2, kNaN2, kNaN2, kNaN2);
            }
            if (i0 == 0 || i0 + P >= nb) {
                // the column's first and last vectors, element by element
#pragma unroll
                for (int v = 0; v < kLoads; ++v) {
                    const int64_t j = jf + (int64_t)(i0 + v / U) * B + (v % U) * 512 + t;
                    if (i0 + v / U < nb && j <= jl && (j == jf || j == jl || j < r.jlo || j >= r.jhi))
                        q[v] = load_edge(r.buf, j, r.mis, cb, ce);
                }
            }
#pragma unroll
            for (int p = 0; p < P; ++p) {
                if (i0 + p >= nb) break;
                uint32_t m = kNaN2;
#pragma unroll
                for (int u = 0; u < U; ++u) m = bmax2(m, vmax(q[p * U + u]));
                s.keys[i0 + p][t] = (uint16_t)key_of(m);
            }
        }
        finish_column<U, true>(a, r, c, false, s);
    }
}

// ---- column mode with finishing warps ----------------------------------------
//
// For rounds with several columns per CTA: warps 0 .. kStreamWarps-1 stream
// (one key slot a thread, two batches of eight loads per thread in
// flight), the other warps finish, one column behind.  The streamers write a column's group keys into
// one of two shared-memory buffers and arrive on its "full" barrier; the
// finishing warps wait there, finish the column from the buffer while the
// streamers fill the other one, and arrive on the buffer's "free" barrier,
// which the streamers wait on before they fill it again.  A column's finish
// then costs no stream time as long as the CTA has columns left to stream.

// The split of a CTA's warps in this mode: SW stream, the others finish.
template <int SW>
struct Team {
    static constexpr int kStreamWarps = SW;
    static constexpr int kStreamThreads = SW * 32;                      // key slots of a batch
    static constexpr int kFinWarps = kWarps - SW;
    static constexpr int kFinThreads = kFinWarps * 32;
    static constexpr int kSlotsPer = kStreamThreads / kFinThreads;      // slots per finishing thread
    static constexpr int kTeamRows = 64 / kSlotsPer < 24 ? 64 / kSlotsPer : 24;   // batches of a column at most
    static constexpr int kSecThreads = kFinThreads / 64;                // finishing threads a section
    static_assert(kSlotsPer * kFinThreads == kStreamThreads && kSlotsPer * kTeamRows <= 64, "slot masks");
    static_assert(kSecThreads * 64 == kFinThreads && kStreamThreads <= 512, "sections, slot ids in 9 bits");
    static_assert(2 * kTeamRows * kStreamThreads <= kKeyRows * 512, "the two key buffers fit in s.keys");
};
constexpr int kBarTeam = 1, kBarFree = 2, kBarFull = 4;     // named barriers (free and full: + buffer)

__device__ __forceinline__ void bar_sync_id(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }
__device__ __forceinline__ void bar_arrive_id(int id, int n) { asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory"); }

// Key buffer b: [batch][slot].
template <int SW>
__device__ __forceinline__ uint16_t *team_keys(Smem &s, int b)
{
    using TM = Team<SW>;
    return &s.keys[0][0] + (size_t)b * TM::kTeamRows * TM::kStreamThreads;
}

// The streamers' part: every column of [c0, c1), one after the other.
template <int U, int SW>
__device__ __forceinline__ void team_stream(const GmRun &r, int64_t c0, int64_t c1, Smem &s)
{
    using TM = Team<SW>;
    constexpr int64_t B = (int64_t)TM::kStreamThreads * U;
    constexpr int P = 16 / U;   // batches a step
    const int st = threadIdx.x;
    for (int64_t c = c0; c < c1; ++c) {
        const int n = (int)(c - c0), b = n & 1;
        if (n >= 2) bar_sync_id(kBarFree + b, kThreads);   // the finishing warps are done with buffer b
        uint16_t *keys = team_keys<SW>(s, b);
        const int64_t cb = c * r.V, ce = cb + r.V;
        const int64_t jf = (cb + r.mis) >> 3, jl = (ce - 1 + r.mis) >> 3;
        const int nb = (int)((jl - jf) / B + 1);
        for (int i0 = 0; i0 < nb; i0 += P) {
            uint4 q[16];
#pragma unroll
            for (int v = 0; v < 16; ++v) {
                const int64_t j = jf + (int64_t)(i0 + v / U) * B + (v % U) * TM::kStreamThreads + st;
                q[v] = (i0 + v / U < nb && j > jf && j < jl && j >= r.jlo && j < r.jhi)
                           ? __ldg(r.vb + j) : make_uint4(kNaN2, kNaN2, kNaN2, kNaN2);
            }
            if (i0 == 0 || i0 + P >= nb) {
                // the column's first and last vectors, element by element
#pragma unroll
                for (int v = 0; v < 16; ++v) {
                    const int64_t j = jf + (int64_t)(i0 + v / U) * B + (v % U) * TM::kStreamThreads + st;
                    if (i0 + v / U < nb && j <= jl && (j == jf || j == jl || j < r.jlo || j >= r.jhi))
                        q[v] = load_edge(r.buf, j, r.mis, cb, ce);
                }
            }
#pragma unroll
            for (int p = 0; p < P; ++p) {
                if (i0 + p >= nb) break;
                uint32_t m = kNaN2;
#pragma unroll
                for (int u = 0; u < U; ++u) m = bmax2(m, vmax(q[p * U + u]));
                keys[(i0 + p) * TM::kStreamThreads + st] = (uint16_t)key_of(m);
            }
        }
        bar_arrive_id(kBarFull + b, kThreads);   // buffer b holds column c's keys
    }
}

// Append the groups of a finishing thread's slots in above and tie (bit
// TM::kTeamRows q + i: batch i of slot ft + TM::kFinThreads q) to the two group
// lists, one shared atomic per warp on the packed count (as append_groups).
template <int SW>
__device__ __forceinline__ void team_append_groups(Smem &s, unsigned long long above, unsigned long long tie, int ft,
                                                   int lane)
{
    using TM = Team<SW>;
    int total;
    const int excl = warp_exclusive_sum(__popcll(above) | (__popcll(tie) << 16), lane, total);
    if (total == 0) return;
    uint32_t base = 0;
    if (lane == 0) base = atomicAdd(&s.ngrp, (uint32_t)total);
    base = __shfl_sync(kFull, base, 0) + (uint32_t)excl;
    uint32_t pa = base & 0xFFFFu, pt = base >> 16;
    for (unsigned long long m = above; m; m &= m - 1, ++pa) {
        const int k = __ffsll((long long)m) - 1;
        if (pa < (uint32_t)kGroupCap)
            s.grp[pa] = ((uint32_t)(k % TM::kTeamRows) << 9) | (uint32_t)(ft + TM::kFinThreads * (k / TM::kTeamRows));
    }
    for (unsigned long long m = tie; m; m &= m - 1, ++pt) {
        const int k = __ffsll((long long)m) - 1;
        if (pt < (uint32_t)kGroupCap)
            s.tgrp[pt] = ((uint32_t)(k % TM::kTeamRows) << 9) | (uint32_t)(ft + TM::kFinThreads * (k / TM::kTeamRows));
    }
}

// The finishing warps' part for column c, whose keys are in buffer b:
// phase 2 as in select_candidates and rank_emit, by TM::kFinThreads threads of
// TM::kSlotsPer key slots each (64 sections of TM::kSecThreads threads), on named
// barrier 1.
template <int U, int SW>
__device__ __forceinline__ void team_finish(const RoundArgs &a, const GmRun &r, int64_t c, int b, Smem &s)
{
    using TM = Team<SW>;
    constexpr int64_t B = (int64_t)TM::kStreamThreads * U;
    constexpr int NW = TM::kFinWarps, BAR = kBarTeam;
    const int ft = threadIdx.x - TM::kStreamThreads, lane = ft & 31, w = ft >> 5;
    const int kk = r.kk;
    const int64_t cb = c * r.V, ce = cb + r.V;
    const int64_t jf = (cb + r.mis) >> 3, jl = (ce - 1 + r.mis) >> 3;
    const int nb = (int)((jl - jf) / B + 1);
    const uint16_t *keys = team_keys<SW>(s, b);
    const RunView rv = view_of(r);
    int32_t draft_tok = -2;   // (thread 0) a target column's draft token; -2: none
    if (!r.draft && ft == 0) {
        const int gp1 = a.gamma + 1;
        const int64_t ln = udiv(c, gp1);
        const int j = (int)(c - ln * gp1);
        if (j < a.gamma) draft_tok = __ldg(a.drafts + ln * a.gamma + j);
    }
    if (ft < kKeyRows) s.tiecnt[ft] = 0u;
    // 1. this thread's slots: their maxima
    uint32_t ms[TM::kSlotsPer], mt = 0;
#pragma unroll
    for (int q = 0; q < TM::kSlotsPer; ++q) {
        ms[q] = 0;
        for (int i = 0; i < nb; ++i) {
            const uint32_t key = keys[i * TM::kStreamThreads + ft + TM::kFinThreads * q];
            ms[q] = key > ms[q] ? key : ms[q];
        }
        mt = ms[q] > mt ? ms[q] : mt;
    }
    // 2. the bound: the kk-th largest of 64 section maxima (kk <= 8) or of
    //    the slot maxima
    uint32_t msec = mt;
#pragma unroll
    for (int d = 1; d < TM::kSecThreads; d <<= 1) {
        const uint32_t o = __shfl_xor_sync(kFull, msec, d);
        msec = o > msec ? o : msec;
    }
    if ((lane & (TM::kSecThreads - 1)) == 0) s.sec[ft / TM::kSecThreads] = msec;
#pragma unroll
    for (int q = 0; q < TM::kSlotsPer; ++q) s.smax[ft + TM::kFinThreads * q] = ms[q];
    team_sync<NW, BAR>();
    const uint32_t T = kk <= 8 ? kth_of_64(s.sec[lane], s.sec[lane + 32], kk)
                               : kth_of_smem(s.smax, TM::kStreamThreads, kk, lane);
    // 3. the groups above T and at it (bit TM::kTeamRows q + i: batch i of slot q)
    unsigned long long above = 0ull, tie = 0ull;
#pragma unroll
    for (int q = 0; q < TM::kSlotsPer; ++q)
        if (ms[q] != 0 && ms[q] >= T)
            for (int i = 0; i < nb; ++i) {
                const uint32_t key = keys[i * TM::kStreamThreads + ft + TM::kFinThreads * q];
                above |= (unsigned long long)(key != 0 && key > T) << (TM::kTeamRows * q + i);
                tie |= (unsigned long long)(key != 0 && key == T) << (TM::kTeamRows * q + i);
            }
    team_append_groups<SW>(s, above, tie, ft, lane);
    team_sync<NW, BAR>();
    if (r.id_map == nullptr && (s.ngrp >> 16) > (uint32_t)kFewTies) {
        // many ties: groups at T per batch; again, from the first batches holding kk
#pragma unroll 1
        for (int i = 0; i < nb; ++i) {
            uint32_t ni = 0;
#pragma unroll
            for (int q = 0; q < TM::kSlotsPer; ++q)
                ni += (uint32_t)__popc(__ballot_sync(kFull, (tie >> (TM::kTeamRows * q + i)) & 1ull));
            if (lane == 0 && ni) atomicAdd(&s.tiecnt[i], ni);
        }
        team_sync<NW, BAR>();
        int acc = 0, upto = TM::kTeamRows;
        for (int i = 0; i < nb; ++i) {
            acc += (int)s.tiecnt[i];
            if (acc >= kk) {
                upto = i + 1;
                break;
            }
        }
        const uint32_t keep_above = s.ngrp & 0xFFFFu;
        team_sync<NW, BAR>();
        if (ft == 0) s.ngrp = keep_above;
        team_sync<NW, BAR>();
        const unsigned long long rows = (1ull << upto) - 1ull;   // upto <= TM::kTeamRows <= 24
        unsigned long long keep = 0ull;
#pragma unroll
        for (int q = 0; q < TM::kSlotsPer; ++q) keep |= rows << (TM::kTeamRows * q);
        team_append_groups<SW>(s, 0ull, tie & keep, ft, lane);
        team_sync<NW, BAR>();
    }
    const int na = (int)(s.ngrp & 0xFFFFu), nt = (int)(s.ngrp >> 16);
    const bool lost = na > kGroupCap || nt > kGroupCap;
    // 4. their elements >= T: one 16-byte vector per thread per pass, four
    //    passes' loads in flight
    if (!lost) {
        const int nv = (na + nt) * U;
        for (int p0 = 0; p0 < nv; p0 += 4 * TM::kFinThreads) {
            uint4 qv[4];
            int64_t jv[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const int p = p0 + h * TM::kFinThreads + ft;
                qv[h] = make_uint4(kNaN2, kNaN2, kNaN2, kNaN2);
                jv[h] = 0;
                if (p < nv) {
                    const uint32_t gid = p / U < na ? s.grp[p / U] : s.tgrp[p / U - na];
                    jv[h] = jf + (int64_t)(gid >> 9) * B + (p % U) * TM::kStreamThreads + (gid & 511u);
                    if (jv[h] < r.NV) qv[h] = load_col_vec(rv, jv[h], cb, ce);
                }
            }
#pragma unroll 1
            for (int h = 0; h < 4; ++h) {
                if (p0 + h * TM::kFinThreads + 32 * w >= nv) break;   // this warp has no vector in the pass
                const uint4 q = h == 0 ? qv[0] : h == 1 ? qv[1] : h == 2 ? qv[2] : qv[3];
                const int64_t j = h == 0 ? jv[0] : h == 1 ? jv[1] : h == 2 ? jv[2] : jv[3];
                uint32_t mask = 0;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const uint32_t key = order_key(half_of(q, e));
                    mask |= (key != 0 && key >= T) ? 1u << e : 0u;
                }
                int total;
                const int excl = warp_exclusive_sum(__popc(mask), lane, total);
                if (total == 0) continue;
                uint32_t pos = 0;
                if (lane == 0) pos = atomicAdd(&s.ncand, (uint32_t)total);
                pos = __shfl_sync(kFull, pos, 0) + (uint32_t)excl;
                for (uint32_t m = mask; m; m &= m - 1, ++pos) {
                    const int e = __ffs(m) - 1;
                    const uint32_t raw = half_of(q, e);
                    uint32_t id = (uint32_t)(8 * j - r.mis - cb + e);
                    if (r.id_map) id = (uint32_t)__ldg(r.id_map + id);
                    if (pos < (uint32_t)kCap) s.cand[pos] = make_entry(order_key(raw), id, raw);
                }
            }
        }
    }
    team_sync<NW, BAR>();
    // 5. the kk best, in order
    const int n = (int)s.ncand;
    if (lost || n > kCap) {
        exact_scan<NW, BAR>(rv, cb, ce, cb, T, s, lane, w);
    } else if (n > kRankMax) {
        select_many<NW, BAR>(n, kk, s, lane, w);
    } else {
        rank_into_list(s, n, kk, ft, TM::kFinThreads);
    }
    team_sync<NW, BAR>();
    if (r.draft) {
        for (int i = ft; i < kk; i += TM::kFinThreads) {
            const unsigned long long e = s.wl[0][i];
            a.out_vals[c * kk + i] = entry_raw(e);
            a.out_ids[c * kk + i] = (int32_t)entry_id(e);
        }
    } else if (w == 0) {
        int32_t token = (int32_t)entry_id(s.wl[0][0]);
        bool accepted;
        if (a.uniforms) accepted = sampled_decide(a, c, s.wl[0], kk, lane, token);
        else accepted = __shfl_sync(kFull, draft_tok, 0) == token;
        lane_done(a, c, token, accepted, lane);
    }
    if (ft == 0) {
        s.ncand = 0u;
        s.ngrp = 0u;
    }
    team_sync<NW, BAR>();
}

// The finishing warps' part: every column of [c0, c1), one column behind
// the streamers.
template <int U, int SW>
__device__ __forceinline__ void team_finish_all(const RoundArgs &a, const GmRun &r, int64_t c0, int64_t c1, Smem &s)
{
    using TM = Team<SW>;
    if (threadIdx.x == TM::kStreamThreads) {
        s.ncand = 0u;
        s.ngrp = 0u;
    }
    team_sync<TM::kFinWarps, kBarTeam>();
    for (int64_t c = c0; c < c1; ++c) {
        const int n = (int)(c - c0), b = n & 1;
        bar_sync_id(kBarFull + b, kThreads);   // buffer b holds column c's keys
        team_finish<U, SW>(a, r, c, b, s);
        if (c + 2 < c1) bar_arrive_id(kBarFree + b, kThreads);   // the streamers may fill buffer b again
    }
}

// ---- one pass: every CTA's slice in its registers ---------------------------
//
// Rounds small enough for each CTA's slice to fit in its registers at once
// (at most 512 L vectors, L loads per thread).  The CTAs of a run are dealt
// out to its columns, as evenly as they go (each column at least one), and
// a column's CTAs split its vectors evenly: CTA b of W works on column
// floor(b cols / W).  A CTA loads its slice, then selects the top-kk of it
// by itself: the bound over its own section (or thread) maxima, its
// elements that reach it.  No group key goes to global memory and nothing
// is read twice.  A column with one CTA is finished right there; otherwise
// every CTA publishes its candidates (at most 2 kk, else its ranked top-kk)
// and the one that takes the column's ticket last merges them -- or, with
// a thread-block cluster per column (MODE 7), the first CTA of the cluster
// merges them from its own shared memory.  Greedy verify publishes one
// argmax entry per CTA and verifies a lane in one step.

// The candidates of the part of a column held by this CTA's slice (vectors
// j0 + u 512 + t in q[u], every element outside the part already the mask
// value; cb the column's first element): its elements that reach the bound
// T, unranked, in s.cand; returns how many (more than kCap: only the first
// kCap kept).  With kk = 1 and no id map, just the part's best element
// (none for an empty part).  Every thread calls it.  Positions inside the
// slice are counted from its vector j0's first element, e0 = 8 j0 - mis, in
// 32 bits.  The code is kept short (rolled loops over the few vectors that
// matter): it runs once per launch, so each new stretch of it is an
// instruction-cache miss.
template <int L>
__device__ __forceinline__ int pass_cands(const GmRun &r, const uint4 (&q)[L], int64_t j0, int64_t cb, Smem &s,
                                          uint32_t &T_out)
{
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const int kk = r.kk;
    const int idb = (int)(8 * j0 - r.mis - cb);   // id of position 0
    // 1. the key of every vector's maximum, two to a word, and this
    //    thread's maximum
    uint32_t vk[(L + 1) / 2];
    uint32_t mt = 0;
#pragma unroll
    for (int u = 0; u < L; ++u) {
        const uint32_t key = key_of(vmax(q[u]));
        mt = key > mt ? key : mt;
        if (u & 1) vk[u >> 1] |= key << 16;
        else vk[u >> 1] = key;
    }
    // 2. the bound T: the kk-th largest section maximum (kk <= 8) or thread
    //    maximum (larger kk, or a part in fewer than kk sections); 0 when
    //    fewer than kk threads hold an element of the part -- then every
    //    element is a candidate, and there are fewer than 8 kk
    uint32_t m8 = mt;
#pragma unroll
    for (int d = 1; d < 8; d <<= 1) {
        const uint32_t o = __shfl_xor_sync(kFull, m8, d);
        m8 = o > m8 ? o : m8;
    }
    if ((lane & 7) == 0) s.sec[4 * w + (lane >> 3)] = m8;
    s.smax[t] = mt;
    if (t == 0) s.last[1] = 0xFFFFFFFFu;   // kk = 1: the shared minimum below
    __syncthreads();
    uint32_t T = kk <= 8 ? kth_of_64(s.sec[lane], s.sec[lane + 32], kk) : 0u;
    if (T == 0u) T = kth_of_smem(s.smax, kThreads, kk, lane);
    T_out = T;
    // the vectors whose maximum reaches T (one or two, mostly)
    uint32_t um = 0;
#pragma unroll
    for (int u = 0; u < L; ++u) {
        const uint32_t key = (vk[u >> 1] >> (16 * (u & 1))) & 0xFFFFu;
        um |= (key != 0 && key >= T) ? 1u << u : 0u;
    }
    if (kk == 1 && r.id_map == nullptr) {
        // the maximum T; of the elements at it, the one with the smallest
        // position (the smallest id: no id map): each thread holding T
        // offers its first (its vectors are in position order), a shared
        // minimum picks among them
        if (um) {
            const int u = __ffs(um) - 1;
            const uint4 v = pick(q, u);
            int e = 7;
#pragma unroll 1
            for (int i = 6; i >= 0; --i)
                if (order_key(half_of(v, i)) == T) e = i;
            atomicMin(&s.last[1], (uint32_t)(8 * (u * 512 + t) + e));
        }
        __syncthreads();
        const uint32_t p = s.last[1];
        if (p == 0xFFFFFFFFu) return 0;
        // the thread holding position p = 8 (u 512 + t) + e writes its entry
        if ((int)((p >> 3) & 511u) == t) {
            const uint32_t raw = half_of(pick(q, (int)(p >> 12)), (int)(p & 7u));
            s.cand[0] = make_entry(T, (uint32_t)((int)p + idb), raw);
        }
        __syncthreads();
        return 1;
    }
    // 3. the candidates: the elements >= T of those vectors, each by the
    //    thread holding it, straight from its registers
#pragma unroll 1
    for (; um; um &= um - 1) {
        const int u = __ffs(um) - 1;
        const uint4 v = pick(q, u);
        const int g0 = 8 * (u * 512 + t);
#pragma unroll 1
        for (int e = 0; e < 8; ++e) {
            const uint32_t raw = half_of(v, e);
            const uint32_t ke = order_key(raw);
            if (ke != 0 && ke >= T) {
                uint32_t id = (uint32_t)(g0 + e + idb);
                if (r.id_map) id = (uint32_t)__ldg(r.id_map + id);
                const uint32_t pos = atomicAdd(&s.ncand, 1u);
                if (pos < (uint32_t)kCap) s.cand[pos] = make_entry(ke, id, raw);
            }
        }
    }
    __syncthreads();
    return (int)s.ncand;
}

// The part's sorted top-kk from its n candidates (pass_cands; bound T),
// into s.wl[0]; returns its length, min(n, kk).  Many candidates: sorted
// lists per warp; more than the buffer holds (massive ties): the part
// [lo, hi) scanned exactly.  Every thread calls it.
__device__ __forceinline__ int pass_rank(const GmRun &r, int n, int64_t cb, int64_t lo, int64_t hi, uint32_t T,
                                         Smem &s)
{
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const int kk = r.kk;
    if (n > kCap) {
        exact_scan<kWarps, 0>(view_of(r), lo, hi, cb, T, s, lane, w);
    } else if (n > kRankMax) {
        select_many<kWarps, 0>(n, kk, s, lane, w);
    } else {
        rank_into_list(s, n, kk, t, kThreads);
    }
    __syncthreads();
    return n < kk ? n : kk;
}

// Column c's list, s.wl[0][0 .. kk), to its outputs (draft) or to verify
// (target; draft_tok: thread 0's copy of the column's draft token, -2 for
// the bonus position).  Every thread calls it.
__device__ __forceinline__ void pass_emit(const RoundArgs &a, const GmRun &r, int64_t c, int32_t draft_tok, Smem &s)
{
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const int kk = r.kk;
    if (r.draft) {
        for (int i = t; i < kk; i += kThreads) {
            const unsigned long long e = s.wl[0][i];
            a.out_vals[c * kk + i] = entry_raw(e);
            a.out_ids[c * kk + i] = (int32_t)entry_id(e);
        }
    } else if (w == 0) {
        int32_t token = (int32_t)entry_id(s.wl[0][0]);
        bool accepted;
        if (a.uniforms) accepted = sampled_decide(a, c, s.wl[0], kk, lane, token);
        else accepted = __shfl_sync(kFull, draft_tok, 0) == token;
        lane_done(a, c, token, accepted, lane);
    }
}

// The CTA that came last to column c (its nc CTAs: units u0, u0 + 1, ...):
// every CTA's published entries (per of them each, 0 for none; the part's
// top-kk or all its candidates), merged, then emitted; the ticket cleared
// for the next launch.  At most kCap entries in all.
__device__ __forceinline__ void pass_merge(const RoundArgs &a, const GmRun &r, int64_t c, int64_t u0, int nc, int per,
                                           int32_t draft_tok, Smem &s)
{
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const int kk = r.kk;
    const int n_all = nc * per;
    for (int i0 = 0; i0 < n_all; i0 += kThreads) {
        const int i = i0 + t;
        const unsigned long long e = i < n_all ? __ldcg(a.partials + (u0 + i / per) * a.pstride + i % per) : 0ull;
        const uint32_t bal = __ballot_sync(kFull, e != 0ull);
        if (bal) {
            uint32_t base = 0;
            if (lane == 0) base = atomicAdd(&s.ncand, (uint32_t)__popc(bal));
            base = __shfl_sync(kFull, base, 0);
            const uint32_t pos = base + (uint32_t)__popc(bal & lanemask_lt());
            if (e != 0ull && pos < (uint32_t)kCap) s.cand[pos] = e;
        }
    }
    __syncthreads();
    const int n = (int)s.ncand < kCap ? (int)s.ncand : kCap;
    if (n > kRankMax) select_many<kWarps, 0>(n, kk, s, lane, w);
    else rank_into_list(s, n, kk, t, kThreads);
    __syncthreads();
    if (t == 0) r.ticket[c] = 0u;   // ready for the next launch
    pass_emit(a, r, c, draft_tok, s);
}

// Greedy verify in one pass: every CTA of a lane's target columns publishes
// its part's best entry (value desc, id asc; 0 for none) and takes the
// lane's ticket (the ticket of the lane's first column); the last of them
// takes each column's best over its CTAs -- the column's argmax -- and
// verifies the lane: the accept length is the number of leading drafts
// equal to their column's argmax, the commit ids those argmaxes up to and
// including position acc, -1 after.  dr: lane j of warp 0 holds draft j
// (early).  Every thread calls it.
__device__ __forceinline__ void pass_lane(const RoundArgs &a, const GmRun &r, int bi, int64_t c,
                                          unsigned long long best, int32_t dr, Smem &s)
{
    const int t = threadIdx.x, lane = t & 31;
    const int gamma = a.gamma, gp1 = gamma + 1;
    const int64_t cols = r.cols;
    const int64_t ln = udiv(c, gp1), cf = ln * gp1;
    const int64_t uf = udiv(cf * r.W + cols - 1, cols);        // the lane's first CTA
    const int nu = (int)(udiv((cf + gp1) * r.W + cols - 1, cols) - uf);
    unsigned long long *pl = a.partials + (int64_t)a.d_units * a.pstride;
    if (t == 0) {
        __stcg(pl + (int64_t)bi * a.pstride, best);
        s.last[0] = atom_add_acq_rel(r.ticket + cf, 1u) == (uint32_t)(nu - 1) ? 1u : 0u;
    }
    if (t < 16) s.wl[1][t] = 0ull;
    __syncthreads();
    if (s.last[0] == 0u) return;
    for (int i = t; i < nu; i += kThreads) {
        const int64_t u = uf + i;
        const unsigned long long e = u == bi ? best : __ldcg(pl + u * a.pstride);
        atomicMax(&s.wl[1][udiv(u * cols, r.W) - cf], e);   // the CTA's column, within the lane
    }
    __syncthreads();
    if (t < 32) {
        const int32_t token = lane < gp1 ? (int32_t)entry_id(s.wl[1][lane]) : -1;
        const uint32_t miss = __ballot_sync(kFull, lane < gamma && dr != token);
        const int acc = miss ? __ffs(miss) - 1 : gamma;
        if (lane < gp1) a.out_commit[ln * gp1 + lane] = lane <= acc ? token : -1;
        count_lane(a.counters, gamma, acc, lane);
        if (lane == 0) {
            a.out_accept[ln] = acc;
            r.ticket[cf] = 0u;   // ready for the next launch
        }
    }
}

// ---- one pass in thread-block clusters (MODE 7) -------------------------------
//
// The same one pass with each column's CTAs (Q of them, all the column has)
// launched as one thread-block cluster: instead of publishing to global
// memory and meeting through a ticket, a column's CTAs store their entries
// straight into the shared memory of the cluster's first CTA and meet at a
// cluster barrier -- no L2 round trip for the merge.  The barriers are the
// hardware's: every CTA of a cluster is resident at once, and every thread
// of every CTA passes both phases.

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_arrive_relaxed() { asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
// the address of this CTA's shared variable p in the CTA of the given rank
__device__ __forceinline__ uint32_t cluster_map(const void *p, uint32_t rank)
{
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
    return a;
}
__device__ __forceinline__ void st_cluster_u64(uint32_t addr, unsigned long long v)
{
    asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}

// The receive area of the cluster's first CTA: per entries from each of the
// Q CTAs, in its group-key buffer (which the one-pass mode does not use).
__device__ __forceinline__ unsigned long long *cluster_inbox(Smem &s)
{
    return reinterpret_cast<unsigned long long *>(&s.keys[0][0]);
}
static_assert(sizeof(Smem::keys) >= 8 * 2 * SPEC_MAX_K * sizeof(unsigned long long), "inbox of 8 CTAs");

// After pass_cands in a cluster of Q CTAs (one column c): the column's
// entries meet in the first CTA, which merges and emits them (greedy verify:
// the column's argmax, with whether it equals the column's draft, goes to
// the lane's fence-free epilogue, lane_done; dtok: lane j of warp 0 holds
// draft j).  n, T: pass_cands' results; [lo, hi): this CTA's part.
__device__ __forceinline__ void cluster_finish(const RoundArgs &a, const GmRun &r, int64_t c, int n, uint32_t T,
                                               int64_t cb, int64_t lo, int64_t hi, bool greedy, int32_t dtok,
                                               Smem &s)
{
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    const uint32_t rank = cluster_rank();
    const int kk = r.kk, per = greedy ? 1 : 2 * kk;
    unsigned long long *inbox = cluster_inbox(s);
    // this CTA's entries: its candidates when at most per, else its top-kk
    const unsigned long long *src = s.cand;
    int cnt = n;
    if (!greedy && n > per) {
        cnt = pass_rank(r, n, cb, lo, hi, T, s);
        src = s.wl[0];
    }
    cluster_wait();   // every CTA of the cluster has started (phase 1, arrived at entry)
    for (int i = t; i < per; i += kThreads)
        st_cluster_u64(cluster_map(inbox + rank * per + i, 0), i < cnt ? src[i] : 0ull);
    cluster_arrive();
    cluster_wait();   // phase 2: the first CTA holds every entry
    if (rank != 0) return;
    uint32_t Q;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(Q));
    if (greedy) {
        unsigned long long best = 0ull;
        if (t < 32) {
            best = lane < (int)Q ? inbox[lane] : 0ull;
#pragma unroll
            for (int d = 16; d > 0; d >>= 1) {
                const unsigned long long o = __shfl_xor_sync(kFull, best, d);
                best = o > best ? o : best;
            }
        }
        if (t < 32) {
            const int gp1 = a.gamma + 1;
            const int j = (int)(c - udiv(c, gp1) * gp1);   // the column's position in its lane
            const int32_t token = (int32_t)entry_id(best);
            const int32_t dj = __shfl_sync(kFull, dtok, j < 32 ? j : 0);
            lane_done(a, c, token, j < a.gamma && dj == token, lane);
        }
        return;
    }
    // merge: the nonzero entries into s.cand, ranked into s.wl[0], emitted
    if (t == 0) s.ncand = 0u;
    __syncthreads();
    const int n_all = (int)Q * per;
    for (int i0 = 0; i0 < n_all; i0 += kThreads) {
        const int i = i0 + t;
        const unsigned long long e = i < n_all ? inbox[i] : 0ull;
        const uint32_t bal = __ballot_sync(kFull, e != 0ull);
        if (bal) {
            uint32_t base = 0;
            if (lane == 0) base = atomicAdd(&s.ncand, (uint32_t)__popc(bal));
            base = __shfl_sync(kFull, base, 0);
            const uint32_t pos = base + (uint32_t)__popc(bal & lanemask_lt());
            if (e != 0ull && pos < (uint32_t)kCap) s.cand[pos] = e;
        }
    }
    __syncthreads();
    const int m = (int)s.ncand < kCap ? (int)s.ncand : kCap;
    if (m > kRankMax) select_many<kWarps, 0>(m, kk, s, lane, w);
    else rank_into_list(s, m, kk, t, kThreads);
    __syncthreads();
    pass_emit(a, r, c, dtok, s);
}

// One-pass mode, all of it, for CTA bi of run r.  A CTA whose column has
// others publishes its candidates unranked when there are at most 2 kk of
// them (the merging CTA ranks them all), else its ranked top-kk.
template <int L, bool CLUSTER>
__device__ __forceinline__ void one_pass(const RoundArgs &a, const GmRun &r, int bi, Smem &s)
{
    const int t = threadIdx.x;
    if constexpr (CLUSTER) cluster_arrive_relaxed();   // phase 1: this CTA runs
    const int64_t cols = r.cols;
    const int64_t c = udiv((int64_t)bi * cols, r.W);                   // this CTA's column
    const int64_t f = udiv(c * r.W + cols - 1, cols);                  // its first CTA
    const int nc = (int)(udiv((c + 1) * r.W + cols - 1, cols) - f);    // and how many
    const int64_t cb = c * r.V, ce = cb + r.V;
    const int64_t jf = (cb + r.mis) >> 3, nvc = ((ce - 1 + r.mis) >> 3) - jf + 1;
    // the column's vectors split among its CTAs: the first nvc mod nc get
    // one more
    const int64_t per_cta = udiv(nvc, nc), extra = nvc - per_cta * nc, sub = bi - f;
    const int64_t j0 = jf + sub * per_cta + (sub < extra ? sub : extra);
    const int64_t j1 = j0 + per_cta + (sub < extra ? 1 : 0);
    // The part: elements [lo, hi).  Its whole vectors [ja, jb) load as
    // vectors; the (at most two) vectors it shares with the next or previous
    // column, or with the buffer's edge, element by element, the rest of
    // them masked.  Plain (L2-cached) loads, not read-only ones: a
    // read-only load may be issued again at a later use instead of being
    // kept in registers.
    const int64_t e0 = 8 * j0 - r.mis, e1 = 8 * j1 - r.mis;
    const int64_t lo = e0 > cb ? e0 : cb, hi = e1 < ce ? e1 : ce;
    int64_t ja = (lo + r.mis + 7) >> 3, jb = (hi + r.mis) >> 3;
    ja = ja > r.jlo ? ja : r.jlo;
    jb = jb < r.jhi ? jb : r.jhi;
    uint4 q[L];
#pragma unroll
    for (int u = 0; u < L; ++u) {
        const int64_t j = j0 + u * 512 + t;
        q[u] = (j >= ja && j < jb) ? __ldcg(r.vb + j) : make_uint4(kNaN2, kNaN2, kNaN2, kNaN2);
    }
    {
        const int64_t jl = (hi - 1 + r.mis) >> 3;   // the part's last vector; j0 its first
#pragma unroll 1
        for (int k2 = 0; k2 < 2; ++k2) {
            const int64_t j = k2 ? jl : j0;
            if ((k2 && jl == j0) || (j >= ja && j < jb) || (int)((j - j0) & 511) != t) continue;
            const uint4 v = load_edge(r.buf, j, r.mis, lo, hi);
            const int u = (int)((j - j0) >> 9);
#pragma unroll
            for (int i = 0; i < L; ++i)
                if (i == u) q[i] = v;
        }
    }
    // a target column's draft token (thread 0); greedy: the lane's drafts
    // (lane j of warp 0 draft j), early
    const bool greedy = !r.draft && a.uniforms == nullptr;
    int32_t dtok = -2;
    if (!r.draft && t < 32) {
        const int gp1 = a.gamma + 1;
        const int64_t ln = udiv(c, gp1);
        const int j = greedy ? t : (int)(c - ln * gp1);
        if (j < a.gamma && (greedy || t == 0)) dtok = __ldg(a.drafts + ln * a.gamma + j);
    }
    uint32_t T;
    const int n = pass_cands<L>(r, q, j0, cb, s, T);
    if constexpr (CLUSTER) {
        cluster_finish(a, r, c, n, T, cb, lo, hi, greedy, dtok, s);
        return;
    }
    if (greedy) {
        // kk = 1, no id map: n <= 1, the best in s.cand[0]
        pass_lane(a, r, bi, c, n ? s.cand[0] : 0ull, dtok, s);
        return;
    }
    const int per = 2 * r.kk;   // entries a CTA publishes (the slot holds them)
    if (nc == 1 || n > per) {
        const int len = pass_rank(r, n, cb, lo, hi, T, s);
        if (nc == 1) {
            pass_emit(a, r, c, dtok, s);
            return;
        }
        unsigned long long *slot = a.partials + ((r.draft ? 0 : a.d_units) + bi) * a.pstride;
        if (t < per) __stcg(slot + t, t < len ? s.wl[0][t] : 0ull);
    } else {
        unsigned long long *slot = a.partials + ((r.draft ? 0 : a.d_units) + bi) * a.pstride;
        if (t < per) __stcg(slot + t, t < n ? s.cand[t] : 0ull);
    }
    __syncthreads();   // the entries are written (and s.cand, s.wl read)
    if (t == 0) {
        s.ncand = 0u;
        s.last[0] = arrive_at_end(r.ticket + c, (uint32_t)(nc - 1));
    }
    __syncthreads();
    if (s.last[0] != 0u) pass_merge(a, r, c, (r.draft ? 0 : a.d_units) + f, nc, per, dtok, s);
}

// ---- whole columns in thread-block clusters (MODE 8) --------------------------
//
// For rounds with fewer columns than three quarters of the SMs and too many
// vectors for one pass (C3): each column is one cluster of Q CTAs (Q from 2
// to 8, the fewest that keep three quarters of the SMs busy).  CTA q of the
// cluster streams batches [q nb / Q, (q + 1) nb / Q) of the column as
// column mode does, its group keys in its own shared memory, and selects
// that part's top-kk with the same finish (bound, groups, ties cut within
// the part, re-read, rank).  The Q lists then meet in the first CTA's inbox
// -- past the end of Smem -- across a cluster barrier, and the first CTA
// merges and emits them.  No tickets, no keys in global memory.
constexpr size_t kInboxOff = (kSmemBytes + 15) & ~(size_t)15;
constexpr size_t kSmemInboxBytes = kInboxOff + 8 * SPEC_MAX_K * sizeof(unsigned long long);
static_assert(kSmemInboxBytes <= 227 * 1024, "one CTA per SM must fit");

template <int U>
__device__ __forceinline__ void cluster_columns(const RoundArgs &a, const GmRun &r, int bi, Smem &s,
                                                unsigned char *base)
{
    constexpr int64_t B = 512 * U;
    static_assert(U == 8, "one batch per step");
    const int t = threadIdx.x, lane = t & 31, w = t >> 5;
    cluster_arrive_relaxed();   // phase 1: this CTA runs
    uint32_t Q;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(Q));
    const uint32_t rank = cluster_rank();
    const int kk = r.kk;
    const int64_t c = udiv(bi, Q);
    const int64_t cb = c * r.V, ce = cb + r.V;
    const int64_t jf = (cb + r.mis) >> 3, jl = (ce - 1 + r.mis) >> 3;
    const int nb = (int)((jl - jf) / B + 1);
    const int i_lo = (int)(rank * nb / Q), i_hi = (int)((rank + 1) * nb / Q);
    if (t < kk) s.wl[0][t] = 0ull;   // the part's list: empty slots stay 0
    // the part's batches, as stream_columns streams a column
    for (int i0 = i_lo; i0 < i_hi; ++i0) {
        uint4 q[kLoads];
#pragma unroll
        for (int v = 0; v < kLoads; ++v) {
            const int64_t j = jf + (int64_t)i0 * B + v * 512 + t;
            q[v] = (j > jf && j < jl && j >= r.jlo && j < r.jhi) ? __ldg(r.vb + j)
                                                                  : make_uint4(kNaN2, kNaN2, kNaN2, kNaN2);
        }
        if (i0 == 0 || i0 + 1 >= nb) {
            // the column's first and last vectors, element by element
#pragma unroll
            for (int v = 0; v < kLoads; ++v) {
                const int64_t j = jf + (int64_t)i0 * B + v * 512 + t;
                if (j <= jl && (j == jf || j == jl || j < r.jlo || j >= r.jhi)) q[v] = load_edge(r.buf, j, r.mis, cb, ce);
            }
        }
        uint32_t m = kNaN2;
#pragma unroll
        for (int u = 0; u < U; ++u) m = bmax2(m, vmax(q[u]));
        s.keys[i0 - i_lo][t] = (uint16_t)key_of(m);
    }
    const Sel sel = select_candidates<U, true>(a, r, c, i_hi - i_lo, s, i_lo);
    // the part's top-kk, as rank_emit ranks a column (exactly over the part
    // when the candidates overflow)
    __syncthreads();
    {
        const int n = (int)s.ncand;
        if (sel.lost || n > kCap) {
            const int64_t e0 = 8 * (jf + (int64_t)i_lo * B) - r.mis, e1 = 8 * (jf + (int64_t)i_hi * B) - r.mis;
            exact_scan<kWarps, 0>(view_of(r), e0 > cb ? e0 : cb, e1 < ce ? e1 : ce, cb, sel.T, s, lane, w);
        } else if (n > kRankMax) {
            select_many<kWarps, 0>(n, kk, s, lane, w);
        } else {
            rank_into_list(s, n, kk, t, kThreads);
        }
    }
    __syncthreads();
    unsigned long long *inbox = reinterpret_cast<unsigned long long *>(base + kInboxOff);
    cluster_wait();   // every CTA of the cluster has started (phase 1, arrived at entry)
    if (t < kk) st_cluster_u64(cluster_map(inbox + rank * kk + t, 0), s.wl[0][t]);
    cluster_arrive();
    cluster_wait();   // phase 2: the first CTA holds every list
    if (rank != 0) return;
    // merge: the nonzero entries into s.cand, ranked into s.wl[0]
    if (t == 0) s.ncand = 0u;
    __syncthreads();
    const int n_all = (int)Q * kk;
    {
        const unsigned long long e = t < n_all ? inbox[t] : 0ull;   // n_all <= 8 * 64 = kThreads
        const uint32_t bal = __ballot_sync(kFull, e != 0ull);
        if (bal) {
            uint32_t pos = 0;
            if (lane == 0) pos = atomicAdd(&s.ncand, (uint32_t)__popc(bal));
            pos = __shfl_sync(kFull, pos, 0) + (uint32_t)__popc(bal & lanemask_lt());
            if (e != 0ull) s.cand[pos] = e;
        }
    }
    __syncthreads();
    const int m = (int)s.ncand;
    if (m > kRankMax) select_many<kWarps, 0>(m, kk, s, lane, w);
    else rank_into_list(s, m, kk, t, kThreads);
    __syncthreads();
    if (r.draft) {
        for (int i = t; i < kk; i += kThreads) {
            const unsigned long long e = s.wl[0][i];
            a.out_vals[c * kk + i] = entry_raw(e);
            a.out_ids[c * kk + i] = (int32_t)entry_id(e);
        }
    } else if (w == 0) {
        int32_t token = (int32_t)entry_id(s.wl[0][0]);
        bool accepted;
        if (a.uniforms) accepted = sampled_decide(a, c, s.wl[0], kk, lane, token);
        else accepted = __shfl_sync(kFull, sel.draft_tok, 0) == token;
        lane_done(a, c, token, accepted, lane);
    }
}

// MODE 0: slice mode; 1: column mode; 2 and 3: column mode with finishing
// warps, 12 (2) or 8 (3) of the 16 streaming; 4: one pass, U loads per
// thread; 7: one pass with a cluster of CTAs per column; 8: whole columns,
// a cluster of CTAs per column.
template <int U, int MODE>
__global__ void __launch_bounds__(kThreads, 1) spec_round_kernel(const __grid_constant__ RoundArgs a)
{
    constexpr int P = MODE == 0 ? kLoads / U : 1;
    pdl_launch_dependents();
    pdl_wait();
    extern __shared__ __align__(16) unsigned char smem[];
    Smem &s = *reinterpret_cast<Smem *>(smem);
    const int b = blockIdx.x;
    if (b >= a.d_units + a.t_units) return;
    const bool draft = b < a.d_units;
    const GmRun r = make_run<U>(a, draft);
    const int bi = draft ? b : b - a.d_units;
    if (threadIdx.x == 0) {
        s.ncand = 0u;
        s.ngrp = 0u;
    }
    if constexpr (MODE == 4 || MODE == 7) {
        one_pass<U, MODE == 7>(a, r, bi, s);
        return;
    }
    if constexpr (MODE == 8) {
        cluster_columns<U>(a, r, bi, s, smem);
        return;
    }
    if constexpr (MODE == 1) {
        stream_columns<U>(a, r, bi, s);
        return;
    }
    if constexpr (MODE == 2 || MODE == 3) {
        constexpr int SW = MODE == 2 ? 12 : 8;
        const int64_t cols = r.cols;
        const int64_t c0 = udiv(bi * cols, r.W), c1 = udiv((bi + 1) * cols, r.W);
        if (threadIdx.x < Team<SW>::kStreamThreads) team_stream<U, SW>(r, c0, c1, s);
        else team_finish_all<U, SW>(a, r, c0, c1, s);
        return;
    }
    if constexpr (MODE == 0) {
        const int64_t g0b = slice_lo(r, bi), g1b = slice_lo(r, bi + 1);
        if (g1b <= g0b) return;
        int64_t cn = udiv(elem_lo<U>(r, g0b), r.V) + 1;   // the column after the one in progress
        int64_t cut = cn * r.V;                      // its first element
        const int64_t cl = udiv(elem_hi<U>(r, g1b - 1) - 1, r.V);
        int64_t cdone = cn - 1;      // the first column not yet handled
        int64_t pend = -1;           // a shared column whose ticket this CTA took inside the stream
        uint32_t pend_old = 0;       // (thread 0) that ticket's count before it
        int64_t gb = g0b;
        for (;;) {
            if (gb < g1b) {
                stream_step<U>(r, gb, g1b, cn, cut);
                gb += P;
            }
            const bool ending = gb >= g1b;
            const int64_t upto = ending ? cl + 1 : cn - 1;   // columns below it are complete here
            while (cdone < upto || (ending && pend >= 0)) {
                int64_t c, wf, wl;
                bool fin;
                if (cdone < upto) {
                    c = cdone++;
                    column_owners<U>(r, c, wf, wl);
                    fin = wf == wl;   // the column lies in this slice: finish it now
                    if (!fin) {
                        __syncthreads();   // this CTA's keys of the column are written
                        if (!ending) {
                            // its part here ends inside the slice (the slice's first
                            // column): take the ticket now, read it at the end
                            if (threadIdx.x == 0) pend_old = atom_add_acq_rel(r.ticket + c, 1u);
                            pend = c;
                        } else {
                            if (threadIdx.x == 0) s.last[0] = arrive_at_end(r.ticket + c, (uint32_t)(wl - wf));
                            __syncthreads();
                            fin = s.last[0] != 0u;
                        }
                    }
                } else {
                    c = pend;
                    pend = -1;
                    column_owners<U>(r, c, wf, wl);
                    __syncthreads();
                    if (threadIdx.x == 0) s.last[0] = pend_old == (uint32_t)(wl - wf) ? 1u : 0u;
                    __syncthreads();
                    fin = s.last[0] != 0u;
                }
                if (fin) finish_column<U, false>(a, r, c, wf != wl, s);
                __syncthreads();   // s.last is read by every thread before it is written again
            }
            if (ending) break;
        }
    }
}

}  // namespace gm
