// The per-warp streaming kernel (large rounds): every warp of a full-GPU
// grid owns a contiguous slice of the flat run of logits and streams it
// through its own ring of three 4 KiB stages (bulk copies completing on
// mbarriers), with its own candidate buffer and certificate per column; the
// warps never wait on one another while streaming.  A column split across
// warps is merged by the warp that completes it (ticket); warps on the same
// split column share their best certificate through global memory.  When
// every warp sees megabytes, each warp's own threshold converges fast and
// this independence wins.
#pragma once

#include "common.cuh"

namespace wrp {

constexpr int kWarpsPerCta = 16;
constexpr int kThreads = kWarpsPerCta * 32;
constexpr int kStageVec = 256;                     // 16-byte vectors per warp stage (4 KiB)
constexpr int kLaneVec = kStageVec / 32;           // vectors per lane per stage
constexpr int kStages = 3;                         // per-warp ring depth (12 KiB in flight per warp)
constexpr int kBufCap = 128;                       // per-warp candidate buffer (entries)
constexpr int kMinSliceVec = 2 * kStageVec;        // smallest slice a warp is given

static_assert(kBufCap >= 2 * SPEC_MAX_K && kBufCap % 32 == 0, "a pruned buffer must leave room");

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

// Write a finished column: its best entries (in the buffer, id order) are
// ranked by value; top-k outputs, or for a target column the argmax and, for
// the lane's last column, the prefix match (one lane per position).
__device__ __noinline__ void emit_column(const RoundArgs &a, const Run &r, int64_t c,
                                         unsigned long long *wb, int n, int lane)
{
    const int kk = r.kk;
    for (int i = lane; i < n; i += 32) {
        const unsigned long long e = wb[i];
        int rank = 0;
        for (int j = 0; j < n; ++j) rank += wb[j] > e;
        if (r.draft) {
            a.out_vals[c * kk + rank] = entry_raw(e);
            a.out_ids[c * kk + rank] = (int32_t)entry_id(e);
        } else if (rank == 0 && !a.uniforms) {
            a.out_commit[c] = (int32_t)entry_id(e);   // column c is position c mod (gamma+1) of its lane
        }
    }
    if (r.draft) return;
    if (a.uniforms) {
        // sampled verify needs the list best first: place every entry at its rank
        const unsigned long long e0 = lane < n ? wb[lane] : 0ull, e1 = lane + 32 < n ? wb[lane + 32] : 0ull;
        int r0 = 0, r1 = 0;
        for (int j = 0; j < n; ++j) {
            r0 += wb[j] > e0;
            r1 += wb[j] > e1;
        }
        __syncwarp();
        if (lane < n) wb[r0] = e0;
        if (lane + 32 < n) wb[r1] = e1;
        __syncwarp();
        sampled_column_done(a, c, wb, n, lane);
        return;
    }
    // the lane's ticket counts its finished columns; the warp that finishes
    // the last one reads the argmaxes back and runs the prefix match
    const int gp1 = a.gamma + 1;
    const int64_t ln = udiv(c, gp1);
    __threadfence();
    __syncwarp();
    unsigned last = 0;
    if (lane == 0) last = atomicAdd(a.lane_ticket + ln, 1u) == (unsigned)a.gamma;
    if (!__shfl_sync(kFull, last, 0)) return;
    __threadfence();
    const int32_t tj = lane < gp1 ? __ldcg(a.out_commit + ln * gp1 + lane) : 0;
    const int32_t dj = lane < a.gamma ? __ldg(a.drafts + ln * a.gamma + lane) : 0;
    const uint32_t miss = __ballot_sync(kFull, lane < a.gamma && dj != tj);
    const int acc = miss ? __ffs(miss) - 1 : a.gamma;
    if (lane < gp1 && lane > acc) a.out_commit[ln * gp1 + lane] = -1;
    count_lane(a.counters, a.gamma, acc, lane);
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
    if (cs.n > kk) { const Pruned pq = buf_prune<kBufCap / 32>(wb, cs.n, kk, lane); cs.n = pq.n; cs.own = pq.t; }
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
                const Pruned pq = buf_prune<kBufCap / 32>(wb, kBufCap, kk, lane);
                cs.n = pq.n;
                cs.own = pq.t;
                if (cs.own > cs.cert) cs.cert = cs.own;
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (entry_key(e8[i]) < cs.cert) ok &= ~(1u << i);
            }
        }
    }
    if (cs.n > kk) { const Pruned pq = buf_prune<kBufCap / 32>(wb, cs.n, kk, lane); cs.n = pq.n; cs.own = pq.t; }
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

    int64_t c = udiv(first_elem(r, w), r.V);       // current column
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
                    uint32_t km = key[0];
#pragma unroll
                    for (int g = 1; g < G; ++g) km = key[g] > km ? key[g] : km;
                    seed = __reduce_max_sync(kFull, km);
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
                    const Pruned pq = buf_prune<kBufCap / 32>(wb, kBufCap, kk, lane);
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
                    const Pruned pq = buf_prune<kBufCap / 32>(wb, cs.n, kk, lane);
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
    if (threadIdx.x == 0) s_gave_up = 0u;
    __syncthreads();
    if (gw >= a.d_units + a.t_units) return;
    if (lane == 0) {
        for (int st = 0; st < kStages; ++st) mbar_init(&ws.full[st], 1);
        fence_mbar_init();
    }
    __syncwarp();

    Run r;
    const bool draft = gw < a.d_units;
    r.draft = draft;
    r.buf = draft ? a.draft : a.target;
    r.V = draft ? a.d_V : a.t_V;
    r.N = (draft ? a.d_cols : a.t_cols) * r.V;
    r.W = draft ? a.d_units : a.t_units;
    r.gw0 = draft ? 0 : a.d_units;
    r.kk = draft ? a.k : a.t_k;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(r.buf);
    r.mis = (int)((a0 >> 1) & 7);                       // element phase of buf in 16 B
    r.vb = reinterpret_cast<const uint4 *>(a0 - 2 * (uintptr_t)r.mis);
    r.NV = (r.N + r.mis + 7) >> 3;
    r.jlo = r.mis ? 1 : 0;
    r.jhi = ((r.N + r.mis) & 7) ? r.NV - 1 : r.NV;
    if (r.jhi < r.jlo) r.jhi = r.jlo;
    const int w = gw - r.gw0;
    if (draft) stream_slice<SLOTS, MAPPED>(a, r, w, a.id_map, ws, lane);
    else stream_slice<SLOTS, false>(a, r, w, nullptr, ws, lane);
}

}  // namespace wrp
