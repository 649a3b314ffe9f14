// select.cu -- stage 2: choose the set, emit it in time order.
//
// "Top-k chooses the set; time chooses the order" (AFN-017), Decision and
// Tie handling belongs to membership: the top k = min(G, budget) groups by
// (score descending, group position ascending) form the set -- ties decided
// while choosing membership -- and the set is emitted in ascending position,
// each group expanded to 4 consecutive token IDs, then the raw tail appended.
//
// Scores are compared as order-preserving uint32 keys (float bits,
// sign-folded, -0 folded to +0).  With s* the k-th largest key and
// need = k - #(key > s*), group g is a member iff key > s*, or key == s* and
// fewer than `need` equal keys precede it (the tie rule, applied during
// membership).  Its output slot is #(key > s* before g) + min(need,
// #(key == s* before g)), so the row comes out in ascending position: no sort
// anywhere.
//
// One 1024-thread CTA per query.  Finding s* among all G keys would take
// several radix passes over every key; instead the CTA narrows the field
// first, exactly:
//  1. Per quad of four groups, the largest key: left by the scorer of the
//     same qsa_decode call, or computed here from the scores.  Thread t takes
//     the maximum over its quads t, t + 1024, ... (a "super-block"); with at
//     least k non-empty super-blocks, L = the k-th largest super-block
//     maximum satisfies #(key >= L) >= k, i.e. L <= s*; any smaller L works
//     too, so only its 10 leading bits are searched for.
//  2. Only quads whose maximum is >= L can hold keys >= L: their four scores
//     are re-read and the keys >= L (typically ~1% of G) are gathered, in no
//     particular order, into shared memory.
//  3. s* is found among those candidates -- one per thread, 5 bits per step,
//     all 32 values of the next digit tested at once (radix passes over
//     12-bit digits of (key - L) when there are more than 1024).
//  4. Membership goes into two group bitmaps, key > s* and key == s*; one
//     popcount / prefix-sum pass over the bitmap words then gives every
//     member its place in ascending position, the tie rule included, and
//     the member's own thread writes its four IDs there.
// When the candidates do not fit in shared memory (e.g. when everything
// ties) the CTA takes the plain path -- the same radix select and an ordered
// emission over all G keys read from the scores.
// Below budget (G <= budget) every group is chosen and the row is 0..T-1.
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kBits = 12;           // radix digit width
constexpr int kBins = 1 << kBits;
constexpr int kCandCap = 8192;      // candidates (key, group) held in shared memory
constexpr int kMaxQpt = 16;         // quads per super-block held in registers
constexpr int kMapWords = kMaxQpt * kThreads * 4 / 32;  // group bitmap words of the narrowed path
constexpr int kQuadCap = 2048;      // flagged quads listed in shared memory

struct SelSmem {
    uint32_t hist[kBins];
    uint32_t cand_key[kCandCap];
    int32_t cand_g[kCandCap];
    uint32_t map_gt[kMapWords];  // members with key > s*
    uint32_t map_eq[kMapWords];  // groups with key == s*
    int32_t qlist[kQuadCap];     // flagged quads, in no particular order
    uint64_t warp_tmp[kWarps];
    uint32_t red[kWarps];
    uint32_t red_hi[kWarps], red_lo[kWarps];
    uint32_t mh[3][33];          // rotating histograms of the one-per-thread search
    uint32_t n_cand, n_quad;
    uint32_t found_digit, found_above;
};

// Block-wide exclusive scan of a 64-bit value; *total receives the sum.
__device__ __forceinline__ uint64_t block_excl_scan(uint64_t v, SelSmem &sm, uint64_t *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint64_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sm.warp_tmp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint64_t w = sm.warp_tmp[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint64_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        sm.warp_tmp[lane] = w;  // inclusive prefix over warps
    }
    __syncthreads();
    const uint64_t warp_before = warp == 0 ? 0 : sm.warp_tmp[warp - 1];
    *total = sm.warp_tmp[kWarps - 1];
    const uint64_t r = warp_before + x - v;
    __syncthreads();  // warp_tmp may be reused by the caller
    return r;
}

__device__ __forceinline__ uint32_t block_max(uint32_t v, SelSmem &sm)
{
    v = __reduce_max_sync(0xffffffffu, v);
    if ((threadIdx.x & 31) == 0) sm.red[threadIdx.x >> 5] = v;
    __syncthreads();
    const uint32_t r = __reduce_max_sync(0xffffffffu, sm.red[threadIdx.x & 31]);
    __syncthreads();
    return r;
}

__device__ __forceinline__ uint32_t block_min(uint32_t v, SelSmem &sm)
{
    v = __reduce_min_sync(0xffffffffu, v);
    if ((threadIdx.x & 31) == 0) sm.red[threadIdx.x >> 5] = v;
    __syncthreads();
    const uint32_t r = __reduce_min_sync(0xffffffffu, sm.red[threadIdx.x & 31]);
    __syncthreads();
    return r;
}

// s* = the k-th largest of the n keys key_at(0..n-1), all within [lo, hi],
// n >= k >= 1; need = k - #(key > s*).  Radix passes over 12-bit digits of
// (key - lo), most significant first; lanes holding the same digit add once.
template <typename KeyAt>
__device__ __forceinline__ void kth_largest(KeyAt key_at, int n, uint32_t k, uint32_t lo, uint32_t hi,
                                            SelSmem &sm, uint32_t &thr, uint32_t &need)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t range = hi - lo;
    const int nbits = range == 0 ? 0 : 32 - __clz(range);
    uint32_t prefix = 0, pmask = 0, remaining = k;
    for (int top = nbits; top > 0; top -= kBits) {
        const int lo_bit = max(top - kBits, 0);
        const uint32_t dmask = (1u << (top - lo_bit)) - 1u;
        for (int i = tid; i < kBins; i += kThreads) sm.hist[i] = 0;
        __syncthreads();
        for (int base = warp * 32; base < n; base += kThreads) {
            const int i = base + lane;
            uint32_t bin = 0xffffffffu;
            if (i < n) {
                const uint32_t off = key_at(i) - lo;
                if ((off & pmask) == prefix) bin = (off >> lo_bit) & dmask;
            }
            const uint32_t peers = __match_any_sync(0xffffffffu, bin);
            if (bin != 0xffffffffu && lane == __ffs(peers) - 1) atomicAdd(&sm.hist[bin], uint32_t(__popc(peers)));
        }
        __syncthreads();
        // thread t owns bins NB*t..NB*t+NB-1; above(d) counts the keys in bins > d
        constexpr int NB = kBins / kThreads;
        uint32_t c[NB], mine = 0;
#pragma unroll
        for (int q = 0; q < NB; ++q) {
            c[q] = sm.hist[NB * tid + q];
            mine += c[q];
        }
        uint64_t total;
        const uint64_t below = block_excl_scan(mine, sm, &total);
        uint32_t above = uint32_t(total - below - mine);
#pragma unroll
        for (int q = NB - 1; q >= 0; --q) {
            if (above < remaining && remaining <= above + c[q]) {
                sm.found_digit = uint32_t(NB * tid + q);
                sm.found_above = above;
            }
            above += c[q];
        }
        __syncthreads();
        prefix |= sm.found_digit << lo_bit;
        pmask |= dmask << lo_bit;
        remaining -= sm.found_above;
        __syncthreads();
    }
    thr = lo + prefix;
    need = remaining;
}

// The k-th largest of at most one key per thread (valid == false: none), all
// valid keys within [lo, hi], at least k of them.  Each step settles the next
// 5 bits of the answer at once: with candidates c_w = prefix + (w << shift),
// w = 0..31, a thread's key reaches the first m of them, m computed directly;
// a 33-bin histogram of m gives #(key >= c_w) for every w, and the digit is
// the largest w whose count still reaches k.  After max_steps steps the
// undecided low bits stay 0, so thr is a lower bound of the k-th largest key;
// when every bit is decided it is exact and need = k - #(key > thr).
// One barrier per step: step s fills histogram s mod 3 and clears (s+2) mod 3
// (whose last readers passed this step's barrier), and every warp derives the
// digit itself.  The three histograms are zero on entry, and again once the
// caller has passed one more barrier after the return.
__device__ __forceinline__ bool kth_largest_1pt(bool valid, uint32_t key, uint32_t k, uint32_t lo, uint32_t hi,
                                                int max_steps, SelSmem &sm, uint32_t &thr, uint32_t &need)
{
    const int tid = threadIdx.x, lane = tid & 31;
    const uint32_t off = key - lo;
    const uint32_t range = hi - lo;
    int nb = range == 0 ? 0 : 32 - __clz(range);
    uint32_t prefix = 0;
    int steps = 0;
    for (; nb > 0 && steps < max_steps; ++steps) {
        uint32_t *h = sm.mh[steps % 3];
        const int step = min(5, nb);
        const int shift = nb - step;
        const uint32_t ncand = 1u << step;
        uint32_t m = 0;
        if (valid && off >= prefix) m = min(ncand, ((off - prefix) >> shift) + 1u);
        const uint32_t peers = __match_any_sync(0xffffffffu, m);
        if (m != 0 && lane == __ffs(peers) - 1) atomicAdd(&h[m], uint32_t(__popc(peers)));
        __syncthreads();
        // count(w) = #(m > w) = sum of h[w+1..32]: a suffix sum over the lanes
        uint32_t c = h[lane + 1];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_down_sync(0xffffffffu, c, o);
            if (lane + o < 32) c += y;
        }
        const uint32_t ok = __ballot_sync(0xffffffffu, uint32_t(lane) < ncand && c >= k);
        const uint32_t digit = 31 - __clz(ok);  // bit 0 is always set: count(0) >= k
        if (tid < 33) sm.mh[(steps + 2) % 3][tid] = 0;
        prefix += digit << shift;
        nb = shift;
    }
    thr = lo + prefix;
    const bool exact = nb == 0;
    const uint32_t above = uint32_t(__syncthreads_count(valid && off > prefix));
    if (steps > 0 && tid < 33) sm.mh[(steps - 1) % 3][tid] = 0;  // the last step's histogram
    if (!exact) return false;
    need = k - above;
    return true;
}

// Ordered emission over the n keys key_at(0..n-1) (ascending position): keys
// > thr and the first `need` keys == thr, each as 4 token IDs at its slot.
template <typename KeyAt, typename GroupAt>
__device__ __forceinline__ void emit_in_order(KeyAt key_at, GroupAt group_at, int n, uint32_t thr, uint32_t need,
                                              int k, int32_t *row, uint32_t *err, SelSmem &sm)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int run = ((n + kWarps - 1) / kWarps + 31) & ~31;
    const int w0 = min(n, warp * run);
    const int w1 = min(n, w0 + run);
    uint32_t n_gt = 0, n_eq = 0;
    for (int base = w0; base < w1; base += 32) {
        const int i = base + lane;
        const uint32_t key = i < w1 ? key_at(i) : 0u;
        n_gt += __popc(__ballot_sync(0xffffffffu, i < w1 && key > thr));
        n_eq += __popc(__ballot_sync(0xffffffffu, i < w1 && key == thr));
    }
    uint64_t tot;
    const uint64_t excl = block_excl_scan(lane == 0 ? ((uint64_t(n_eq) << 32) | n_gt) : 0, sm, &tot);
    const uint64_t mine = __shfl_sync(0xffffffffu, excl, 0);  // lane 0 holds the warp's prefix
    uint32_t gt_c = uint32_t(mine);
    uint32_t eq_c = uint32_t(mine >> 32);
    const uint32_t lt_mask = (1u << lane) - 1u;
    for (int base = w0; base < w1; base += 32) {
        const int i = base + lane;
        const uint32_t key = i < w1 ? key_at(i) : 0u;
        const bool is_gt = i < w1 && key > thr;
        const bool is_eq = i < w1 && key == thr;
        const uint32_t bg = __ballot_sync(0xffffffffu, is_gt);
        const uint32_t be = __ballot_sync(0xffffffffu, is_eq);
        const uint32_t my_gt = gt_c + __popc(bg & lt_mask);  // greater keys before this one
        const uint32_t my_eq = eq_c + __popc(be & lt_mask);  // equal keys before this one
        int pos = -1;
        if (is_gt) pos = int(my_gt + min(need, my_eq));
        else if (is_eq && my_eq < need) pos = int(my_gt + my_eq);
        if (pos >= k) {  // cannot happen for a correct threshold; never write past the row
            set_error(err, QSA_DEVERR_ROW_RANGE);
            pos = -1;
        }
        if (pos >= 0) {
            const int g = group_at(i);
            int32_t *o = row + kGroup * pos;
            o[0] = kGroup * g;
            o[1] = kGroup * g + 1;
            o[2] = kGroup * g + 2;
            o[3] = kGroup * g + 3;
        }
        gt_c += __popc(bg);
        eq_c += __popc(be);
    }
}

// The raw scorer's per-SM weights for its next launch, from the times its
// CTAs recorded (run by one spare CTA, after the scorer has finished).  The
// rate of an SM is its tiles over the time of its slower CTA; the weight is
// that rate relative to the mean, x 4096, folded into the weight the SM had
// with a factor 1/4 (the weights converge to the rates without following
// each launch's noise), kept within [1024, 16384].  The
// recorded times are then cleared, so that a launch that records nothing
// leaves the weights as they are.
__device__ void balance_update(ScoreBalance *bl, SelSmem &sm)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool had = __ldcg(&bl->magic) == kBalMagic;
    float rate = 0.0f;
    uint32_t w_old = 0;
    if (tid < kBalSlots) {
        const uint32_t e0 = __ldcg(&bl->el_ns[tid][0]), e1 = __ldcg(&bl->el_ns[tid][1]);
        const uint32_t t0 = __ldcg(&bl->tiles[tid][0]), t1 = __ldcg(&bl->tiles[tid][1]);
        if (e0 > 0u) rate = float(t0 + t1) / float(max(e0, e1));
        w_old = had ? __ldcg(&bl->w[tid]) : 0u;
    }
    float s = rate;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) sm.red[warp] = __float_as_uint(s);
    const int n = __syncthreads_count(rate > 0.0f);
    if (n == 0) return;  // nothing recorded since the last update
    float total = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) total += __uint_as_float(sm.red[w]);
    const float mean = total / float(n);
    uint32_t wn = 0;
    if (rate > 0.0f && mean > 0.0f) {
        const float r = rate / mean * 4096.0f;
        const float u = w_old > 0u ? 0.75f * float(w_old) + 0.25f * r : r;
        wn = uint32_t(fminf(fmaxf(u, 1024.0f), 16384.0f));
    }
    uint64_t tot;
    const uint64_t before = block_excl_scan(wn, sm, &tot);
    if (tid < kBalSlots) {
        bl->w[tid] = wn;
        bl->w_before[tid] = uint32_t(before);
        bl->el_ns[tid][0] = 0u;
        bl->el_ns[tid][1] = 0u;
        bl->tiles[tid][0] = 0u;
        bl->tiles[tid][1] = 0u;
    }
    if (tid == 0) {
        bl->w_total = uint32_t(tot);
        bl->nsm = uint32_t(n);
        bl->magic = kBalMagic;
    }
}

__global__ void __launch_bounds__(kThreads, 1)
select_emit_kernel(const SelectArgs a)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SelSmem &sm = *reinterpret_cast<SelSmem *>(smem_raw);
    const int b = blockIdx.x;
    const int tid = threadIdx.x;
    if (a.bal != nullptr && b == a.batch) {  // the spare CTA: the scorer's next weights
        allow_successor_launch();
        wait_for_predecessor();
        balance_update(a.bal, sm);
        return;
    }
    allow_successor_launch();
    wait_for_predecessor();  // the scores (and quad maxima) come from the previous kernel;
                             // this kernel may start before that one ends, so what it wrote is
                             // read with L2-coherent loads (__ldcg), never the read-only path

    // The quad maxima left by this call's scorer do not depend on T for their
    // address: load them together with T (one round trip instead of two).
    const uint32_t *qmg = a.qmax != nullptr ? a.qmax + int64_t(b) * a.qmax_stride : nullptr;
    uint32_t qv[kMaxQpt];
#pragma unroll
    for (int j = 0; j < kMaxQpt; ++j) {
        const int q = tid + j * kThreads;
        qv[j] = (qmg != nullptr && q < a.qmax_stride) ? __ldcg(qmg + q) : 0u;
    }
    const int T = __ldg(a.visible + b);
    const int32_t *smap = a.slot_map != nullptr ? a.slot_map + __ldg(a.slot_offset + b) : nullptr;
    int32_t *row = a.ids + int64_t(b) * a.row_cap;
    if (T < 0 || T > a.max_visible) {
        if (tid == 0) {
            a.n_ids[b] = 0;
            set_error(a.err, QSA_DEVERR_VISIBLE_RANGE);
        }
        return;
    }
    const int G = T >> 2;
    const int tail = T & 3;
    const int k = G < a.budget ? G : a.budget;
    if (G <= a.budget) {
        // Every complete group is chosen: the row is the dense causal row.
        for (int i = tid; i < T; i += kThreads) row[i] = i;
        if (tid == 0) a.n_ids[b] = T;
        return;
    }

    const float *sc = a.scores + int64_t(b) * a.score_stride;
    auto key_all = [&](int i) -> uint32_t { return order_key(__ldcg(sc + i)); };
    bool done = false;  // (uniform across the CTA)

    // ---- narrowed path: quad maxima -> L <= s* -> candidates -> s* -> bitmap -------
    // Super-block t = the quads t, t + 1024, t + 2048, ... (any partition into
    // disjoint non-empty blocks gives the bound); loads stay coalesced.
    const int nq = (G + 3) / 4;                       // quads of groups
    const int qpt = (nq + kThreads - 1) / kThreads;   // quads per super-block
    const int nsb = min(nq, kThreads);                // non-empty super-blocks
    if (nsb >= k && qpt <= kMaxQpt) {
        const int lane = tid & 31, warp = tid >> 5;
        const int nwords = (G + 31) / 32;
        for (int i = tid; i < nwords; i += kThreads) {
            sm.map_gt[i] = 0u;
            sm.map_eq[i] = 0u;
        }
        if (tid < 3 * 33) sm.mh[tid / 33][tid % 33] = 0u;
        if (tid == 0) {
            sm.n_cand = 0u;
            sm.n_quad = 0u;
        }
#pragma unroll
        for (int j = 0; j < kMaxQpt; ++j) {
            const int q = tid + j * kThreads;
            if (!(j < qpt && q < nq)) {
                qv[j] = 0;
            } else if (qmg == nullptr) {  // no hint: the quad maxima from the scores
                const float4 s4 = __ldcg(reinterpret_cast<const float4 *>(sc + 4 * q));
                uint32_t m = order_key(s4.x);
                if (4 * q + 1 < G) m = max(m, order_key(s4.y));
                if (4 * q + 2 < G) m = max(m, order_key(s4.z));
                if (4 * q + 3 < G) m = max(m, order_key(s4.w));
                qv[j] = m;
            }
        }
        uint32_t sbmax = 0;
#pragma unroll
        for (int j = 0; j < kMaxQpt; ++j) sbmax = max(sbmax, qv[j]);
        const bool has_sb = tid < nsb;
        // range of the super-block maxima: one barrier
        {
            const uint32_t wmx = __reduce_max_sync(0xffffffffu, sbmax);
            const uint32_t wmn = __reduce_min_sync(0xffffffffu, has_sb ? sbmax : 0xffffffffu);
            if (lane == 0) {
                sm.red_hi[warp] = wmx;
                sm.red_lo[warp] = wmn;
            }
        }
        __syncthreads();
        const uint32_t hi = __reduce_max_sync(0xffffffffu, sm.red_hi[lane]);
        const uint32_t lo = __reduce_min_sync(0xffffffffu, sm.red_lo[lane]);
        // L: the 10 leading bits of the k-th largest super-block maximum, the rest 0
        uint32_t L, needL;
        (void)kth_largest_1pt(has_sb, sbmax, uint32_t(k), lo, hi, 2, sm, L, needL);

        // Candidates: the groups with key >= L of the quads whose maximum
        // reaches L, gathered into shared memory in any order.  The flagged
        // quads are listed first (one slot reservation per warp), so that
        // their scores then take a single round of loads, at most
        // kQuadCap / 1024 per thread.
        const uint32_t lt = (1u << lane) - 1u;
        {
            uint32_t bals[kMaxQpt], wtotal = 0;
#pragma unroll
            for (int j = 0; j < kMaxQpt; ++j) {
                bals[j] = __ballot_sync(0xffffffffu, j < qpt && tid + j * kThreads < nq && qv[j] >= L);
                wtotal += __popc(bals[j]);
            }
            uint32_t base = 0;
            if (lane == 0 && wtotal != 0u) base = atomicAdd(&sm.n_quad, wtotal);
            base = __shfl_sync(0xffffffffu, base, 0);
#pragma unroll
            for (int j = 0; j < kMaxQpt; ++j) {
                const uint32_t slot = base + __popc(bals[j] & lt);
                if (((bals[j] >> lane) & 1u) && slot < uint32_t(kQuadCap)) sm.qlist[slot] = tid + j * kThreads;
                base += __popc(bals[j]);
            }
        }
        __syncthreads();
        const uint32_t n_flag = sm.n_quad;
        if (n_flag <= uint32_t(kQuadCap)) {
            constexpr int kPer = kQuadCap / kThreads;  // 2
            int qs[kPer];
            float4 sv[kPer];
#pragma unroll
            for (int f = 0; f < kPer; ++f) {
                const int e = tid + f * kThreads;
                qs[f] = e < int(n_flag) ? sm.qlist[e] : -1;
            }
#pragma unroll
            for (int f = 0; f < kPer; ++f)
                sv[f] = qs[f] >= 0 ? __ldcg(reinterpret_cast<const float4 *>(sc + 4 * qs[f]))
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
            uint32_t keys[kPer][4], cb[kPer][4], wtotal = 0;
#pragma unroll
            for (int f = 0; f < kPer; ++f) {
                const float vals[4] = {sv[f].x, sv[f].y, sv[f].z, sv[f].w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    keys[f][u] = order_key(vals[u]);
                    cb[f][u] = __ballot_sync(0xffffffffu, qs[f] >= 0 && 4 * qs[f] + u < G && keys[f][u] >= L);
                    wtotal += __popc(cb[f][u]);
                }
            }
            uint32_t base = 0;
            if (lane == 0 && wtotal != 0u) base = atomicAdd(&sm.n_cand, wtotal);
            base = __shfl_sync(0xffffffffu, base, 0);
#pragma unroll
            for (int f = 0; f < kPer; ++f) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint32_t slot = base + __popc(cb[f][u] & lt);
                    if (((cb[f][u] >> lane) & 1u) && slot < uint32_t(kCandCap)) {
                        sm.cand_key[slot] = keys[f][u];
                        sm.cand_g[slot] = 4 * qs[f] + u;
                    }
                    base += __popc(cb[f][u]);
                }
            }
        } else if (tid == 0) {
            sm.n_cand = 0u;  // too many flagged quads: the plain path below
        }
        __syncthreads();
        const uint32_t n_c = sm.n_cand;  // published by the barrier above
        if (n_c >= uint32_t(k) && n_c <= uint32_t(kCandCap)) {
            const int n = int(n_c);
            uint32_t thr, need;
            if (n <= kThreads) {
                const bool have = tid < n;
                (void)kth_largest_1pt(have, have ? sm.cand_key[tid] : 0u, uint32_t(k), L, hi, 32, sm, thr, need);
            } else {
                kth_largest([&](int i) { return sm.cand_key[i]; }, n, uint32_t(k), L, hi, sm, thr, need);
            }
            // membership bitmaps; the slot-map line of every possible member
            // (4g < T: inside the query's slot map) is asked of L2 for the
            // attention, which resolves the emitted IDs through it
            for (int i = tid; i < n; i += kThreads) {
                const uint32_t key = sm.cand_key[i];
                const int g = sm.cand_g[i];
                if (key > thr) atomicOr(&sm.map_gt[g >> 5], 1u << (g & 31));
                else if (key == thr) atomicOr(&sm.map_eq[g >> 5], 1u << (g & 31));
                if (smap != nullptr && key >= thr) prefetch_l2(smap + 4 * int64_t(g));
            }
            __syncthreads();
            // Word prefixes: thread t takes the words of groups 64t .. 64t+63;
            // #(key > s*) and #(key == s*) before each word go to shared
            // memory (the radix histogram's space, free by now).
            constexpr int WPT = kMapWords / kThreads;  // 2
            static_assert(2 * kMapWords <= kBins, "word prefixes fit in the histogram space");
            uint32_t *pre_gt = sm.hist, *pre_eq = sm.hist + kMapWords;
            uint32_t wg[WPT], we[WPT], n_gt = 0, n_eq = 0;
#pragma unroll
            for (int w = 0; w < WPT; ++w) {
                const int wi = WPT * tid + w;
                wg[w] = wi < nwords ? sm.map_gt[wi] : 0u;
                we[w] = wi < nwords ? sm.map_eq[wi] : 0u;
                n_gt += __popc(wg[w]);
                n_eq += __popc(we[w]);
            }
            uint64_t tot;
            const uint64_t before = block_excl_scan((uint64_t(n_eq) << 32) | n_gt, sm, &tot);
            uint32_t gt_c = uint32_t(before), eq_c = uint32_t(before >> 32);
#pragma unroll
            for (int w = 0; w < WPT; ++w) {
                pre_gt[WPT * tid + w] = gt_c;
                pre_eq[WPT * tid + w] = eq_c;
                gt_c += __popc(wg[w]);
                eq_c += __popc(we[w]);
            }
            __syncthreads();
            // each member writes its IDs at #(key > s* before it) +
            // min(need, #(key == s* before it)); equal keys past `need` are out
            for (int i = tid; i < n; i += kThreads) {
                const uint32_t key = sm.cand_key[i];
                if (key < thr) continue;
                const int g = sm.cand_g[i];
                const int wi = g >> 5;
                const uint32_t below = (1u << (g & 31)) - 1u;
                const uint32_t gt_b = pre_gt[wi] + __popc(sm.map_gt[wi] & below);
                const uint32_t eq_b = pre_eq[wi] + __popc(sm.map_eq[wi] & below);
                int pos = -1;
                if (key > thr) pos = int(gt_b + min(need, eq_b));
                else if (eq_b < need) pos = int(gt_b + eq_b);
                if (pos >= k) {  // cannot happen for a correct threshold; never write past the row
                    set_error(a.err, QSA_DEVERR_ROW_RANGE);
                    pos = -1;
                }
                if (pos >= 0) {
                    int32_t *o = row + kGroup * pos;
                    o[0] = kGroup * g;
                    o[1] = kGroup * g + 1;
                    o[2] = kGroup * g + 2;
                    o[3] = kGroup * g + 3;
                }
            }
            done = true;
        }
    }

    // ---- plain path: every key ----------------------------------------------------
    if (!done) {
        uint32_t mn = 0xffffffffu, mx = 0;
        for (int i = tid; i < G; i += kThreads) {
            const uint32_t key = key_all(i);
            mn = min(mn, key);
            mx = max(mx, key);
        }
        const uint32_t hi = block_max(mx, sm);
        const uint32_t lo = block_min(mn, sm);
        uint32_t thr, need;
        kth_largest(key_all, G, uint32_t(k), lo, hi, sm, thr, need);
        emit_in_order(key_all, [](int i) { return i; }, G, thr, need, k, row, a.err, sm);
    }
    if (tid < tail) row[kGroup * k + tid] = kGroup * G + tid;
    if (tid == 0) a.n_ids[b] = kGroup * k + tail;
}

}  // namespace

cudaError_t launch_select(const SelectArgs &a, cudaStream_t s, bool pdl)
{
    if (a.batch == 0) return cudaSuccess;
    const size_t smem = sizeof(SelSmem);
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(select_emit_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    const unsigned grid = unsigned(a.batch) + (a.bal != nullptr ? 1u : 0u);
    return launch_kernel(select_emit_kernel, dim3(grid), dim3(kThreads), smem, s, pdl, a);
}

}  // namespace qsa
