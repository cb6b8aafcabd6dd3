// route.cuh -- device helpers of the decode-size kernels: the plan of the
// touched experts, the per-CTA bucketing, top-K selection and the loading of
// token activations.  The CTA-wide helpers take the participating threads'
// index and count and a synchronisation functor, so a kernel whose producer
// warp runs apart can call them on its consumer warps alone.
#pragma once

#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace strata {

struct BlockSync {
    __device__ void operator()() const { __syncthreads(); }
};

// ------------------------------------------------------------------- plan
// A layer's plan: the touched experts in ascending id, their slot ranges,
// and the token of each slot (-1: none).
struct SPlan {
    int n;
    int e[kMaxExperts];
    int off[kMaxExperts];
    int cnt[kMaxExperts];
    int tok[kDecodeMaxTokens * kMaxTopK];
};

__device__ inline void load_plan(SPlan& P, const int32_t* plan, int E, int TK) {
    const int* base = plan + kPlanHeader;
    for (int i = threadIdx.x; i < 3 * E + TK; i += blockDim.x) {
        const int v = __ldcg(base + i);
        if (i < E)
            P.e[i] = v;
        else if (i < 2 * E)
            P.off[i - E] = v;
        else if (i < 3 * E)
            P.cnt[i - 2 * E] = v;
        else
            P.tok[i - 3 * E] = v;
    }
    if (threadIdx.x == 0) P.n = __ldcg(plan);
    __syncthreads();
}

__device__ inline void shared_plan(SPlan& P, int T) {
    for (int s = threadIdx.x; s < T; s += blockDim.x) P.tok[s] = s;
    if (threadIdx.x == 0) {
        P.n = 1;
        P.e[0] = 0;
        P.off[0] = 0;
        P.cnt[0] = T;
    }
    __syncthreads();
}

// Where a bucketing is published (any pointer may be null).
struct BucketOut {
    int32_t* counts;
    int32_t* offsets;
    int32_t* perm;
    int32_t* inv;
    int32_t* plan;
};

// The global copies of a bucketing from the plan P and s_inv (any number of
// pairs; no barrier inside): counts[e], offsets[0..E], perm, inv and the
// plan, as bucket_cta writes them.
__device__ inline void publish_bucket(int TK, int E, const SPlan& P, const int* s_inv,
                                      const BucketOut& g, int tid, int nthr) {
    #pragma unroll 1
    for (int e = tid; e < E; e += nthr) {
        int off = 0, cnt = 0;
        #pragma unroll 1
        for (int u = 0; u < P.n; ++u) {
            off += P.e[u] < e ? P.cnt[u] : 0;
            cnt += P.e[u] == e ? P.cnt[u] : 0;
        }
        if (g.counts) g.counts[e] = cnt;
        if (g.offsets) g.offsets[e] = off;
    }
    if (tid == 0 && g.offsets) {
        int tot = 0;
        for (int u = 0; u < P.n; ++u) tot += P.cnt[u];
        g.offsets[E] = tot;
    }
    #pragma unroll 1
    for (int p = tid; p < TK; p += nthr) {
        const int sl = s_inv[p];
        if (g.inv) g.inv[p] = sl;
        if (g.perm && sl >= 0) g.perm[sl] = p;
    }
    if (g.plan) {
        if (tid == 0) g.plan[0] = P.n;
        #pragma unroll 1
        for (int i = tid; i < P.n; i += nthr) {
            g.plan[kPlanHeader + i] = P.e[i];
            g.plan[kPlanHeader + E + i] = P.off[i];
            g.plan[kPlanHeader + 2 * E + i] = P.cnt[i];
        }
        #pragma unroll 1
        for (int sl = tid; sl < TK; sl += nthr) g.plan[kPlanHeader + 3 * E + sl] = P.tok[sl];
    }
}

// bucket_cta for at most 32 pairs: warp 0 holds pair p in lane p and ranks
// it by (expert, p) with shuffles -- the same slots as the counting sort --
// then one barrier; the global copies (when asked for) follow from P.
template <typename Sync>
__device__ void bucket_warp(const int* s_ids, int TK, int K, int E, SPlan& P, int* s_inv,
                            const BucketOut& g, int tid, int nthr, Sync sync) {
    const int lane = tid & 31;
    if (tid < 32) {
        const int p = lane;
        const int e = p < TK ? s_ids[p] : -1;
        const bool ok = e >= 0 && e < E;
        const int key = ok ? e : 0x7fffffff;          // no slot: ranked after every valid pair
        int rank = 0, before = 0, cnt = 0;
        #pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int kj = __shfl_sync(0xffffffffu, key, j);
            rank += (kj < key || (kj == key && j < p)) ? 1 : 0;
            before += (kj == key && j < p) ? 1 : 0;
            cnt += kj == key ? 1 : 0;
        }
        const bool first = ok && before == 0;        // its expert's first pair
        const unsigned fm = __ballot_sync(0xffffffffu, first);
        int uidx = 0;                                // touched experts below this one
        #pragma unroll
        for (int j = 0; j < 32; ++j) {
            const int kj = __shfl_sync(0xffffffffu, key, j);
            uidx += (((fm >> j) & 1u) != 0u && kj < key) ? 1 : 0;
        }
        const int nvalid = __popc(__ballot_sync(0xffffffffu, ok));
        if (p < TK) s_inv[p] = ok ? rank : -1;
        if (ok) P.tok[rank] = p / K;
        if (first) {
            P.e[uidx] = key;
            P.off[uidx] = rank;
            P.cnt[uidx] = cnt;
        }
        if (nvalid + lane < TK) P.tok[nvalid + lane] = -1;
        if (lane == 0) P.n = __popc(fm);
    }
    sync();
    if (g.counts || g.offsets || g.perm || g.inv || g.plan) {
        publish_bucket(TK, E, P, s_inv, g, tid, nthr);
        sync();
    }
}

// Stable counting sort of the T*K (token, k) pairs by expert, by one CTA.
// s_ids: the pairs' expert ids; an out-of-range id gets no slot (inv -1).
// Fills P and s_inv in shared memory and, when given, the global copies:
// counts[e], offsets[0..E], perm[slot] = t*K + k (slots of one expert in
// ascending t), inv[t*K + k] = slot, and the plan.
template <typename Sync>
__device__ void bucket_cta(const int* s_ids, int T, int K, int E, int* s_cnt, int* s_off,
                           int* s_wsum, SPlan& P, int* s_inv, const BucketOut& g, int tid,
                           int nthr, Sync sync) {
    const int lane = tid & 31, wid = tid >> 5, wpb = nthr >> 5;
    const int TK = T * K;
    if (TK <= 32) {
        bucket_warp(s_ids, TK, K, E, P, s_inv, g, tid, nthr, sync);
        return;
    }
    #pragma unroll 1
    for (int e = tid; e < E; e += nthr) s_cnt[e] = 0;
    #pragma unroll 1
    for (int p = tid; p < TK; p += nthr) s_inv[p] = -1;
    sync();
    #pragma unroll 1
    for (int p = tid; p < TK; p += nthr) {
        const int e = s_ids[p];
        if (e >= 0 && e < E) atomicAdd(&s_cnt[e], 1);
    }
    sync();
    // exclusive scan over experts of (slots, touched experts), packed in one
    // int (slots < 2^16, experts < 2^15); each thread one contiguous segment
    const int seg = (E + nthr - 1) / nthr;
    const int e0 = min(E, tid * seg), e1 = min(E, e0 + seg);
    int local = 0, nz = 0;
    #pragma unroll 1
    for (int e = e0; e < e1; ++e) {
        local += s_cnt[e];
        nz += s_cnt[e] > 0 ? 1 : 0;
    }
    const int mine = local | (nz << 16);
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) s_wsum[wid] = incl;
    sync();
    if (tid == 0) {
        int r = 0;
        #pragma unroll 1
        for (int w = 0; w < wpb; ++w) {
            const int c = s_wsum[w];
            s_wsum[w] = r;
            r += c;
        }
        s_off[E] = r & 0xffff;
        P.n = r >> 16;
    }
    sync();
    const int excl = s_wsum[wid] + incl - mine;
    int run = excl & 0xffff, rank = excl >> 16;
    #pragma unroll 1
    for (int e = e0; e < e1; ++e) {
        s_off[e] = run;
        if (s_cnt[e] > 0) {
            P.e[rank] = e;
            P.off[rank] = run;
            P.cnt[rank] = s_cnt[e];
            ++rank;
        }
        run += s_cnt[e];
    }
    sync();
    #pragma unroll 1
    for (int s = s_off[E] + tid; s < TK; s += nthr) P.tok[s] = -1;
    #pragma unroll 1
    for (int e = tid; e < E; e += nthr) {
        const int c = s_cnt[e];
        if (g.counts) g.counts[e] = c;
        if (g.offsets) g.offsets[e] = s_off[e];
        if (c == 0) continue;
        int slot = s_off[e];
        #pragma unroll 1
        for (int p = 0; p < TK; ++p)
            if (s_ids[p] == e) {
                s_inv[p] = slot;
                P.tok[slot] = p / K;
                if (g.perm) g.perm[slot] = p;
                ++slot;
            }
    }
    sync();
    if (tid == 0 && g.offsets) g.offsets[E] = s_off[E];
    if (g.inv)
        #pragma unroll 1
        for (int p = tid; p < TK; p += nthr) g.inv[p] = s_inv[p];
    if (g.plan) {
        if (tid == 0) g.plan[0] = P.n;
        #pragma unroll 1
        for (int i = tid; i < P.n; i += nthr) {
            g.plan[kPlanHeader + i] = P.e[i];
            g.plan[kPlanHeader + E + i] = P.off[i];
            g.plan[kPlanHeader + 2 * E + i] = P.cnt[i];
        }
        #pragma unroll 1
        for (int s = tid; s < TK; s += nthr) g.plan[kPlanHeader + 3 * E + s] = P.tok[s];
    }
}

// Tail-skip of one call's routing (PolyStrata, "Models and backends",
// section "What was tuned"): an expert that every token of the call ranks
// at place n + 1 or later of its K picks is left out; the picks that stay
// keep their weights.  A pick's place counts its token's picks with a
// larger weight, or an equal weight and a lower id (the selection's order).
// Writes bid[p] = s_ids[p], or -1 for a left-out pick (no slot in the
// bucketing), and sets a left-out pick's weight to 0.  rank: T*K ints,
// keep: E ints of scratch.  Every thread of the CTA calls it.
__device__ inline void tail_skip_cta(const int* s_ids, float* s_w, int T, int K, int E, int n,
                                     int* rank, int* bid, int* keep, int tid, int nthr) {
    const int TK = T * K;
    #pragma unroll 1
    for (int e = tid; e < E; e += nthr) keep[e] = 0;
    #pragma unroll 1
    for (int p = tid; p < TK; p += nthr) {
        const int t0 = (p / K) * K, id = s_ids[p];
        const float w = s_w[p];
        int r = 0;
        #pragma unroll 1
        for (int j = t0; j < t0 + K; ++j) r += (s_w[j] > w || (s_w[j] == w && s_ids[j] < id)) ? 1 : 0;
        rank[p] = r;
    }
    __syncthreads();
    #pragma unroll 1
    for (int p = tid; p < TK; p += nthr) {
        const int id = s_ids[p];
        if (rank[p] < n && id >= 0 && id < E) keep[id] = 1;
    }
    __syncthreads();
    #pragma unroll 1
    for (int p = tid; p < TK; p += nthr) {
        const int id = s_ids[p];
        const bool valid = id >= 0 && id < E;
        const bool left_out = valid && keep[id] == 0;
        bid[p] = valid && !left_out ? id : -1;
        if (left_out) s_w[p] = 0.0f;
    }
    __syncthreads();
}

// ------------------------------------------------------------- selection
// Order-preserving 32-bit key of a logit: a larger float has a larger key.
// NaN (and a taken entry) gets key 0, which never wins.
__device__ __forceinline__ uint32_t logit_key(float v) {
    const uint32_t u = __float_as_uint(v);
    const uint32_t k = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return (v == v) ? k : 0u;
}
__device__ __forceinline__ float key_logit(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Top-K of one token's logits (larger first, ties to the lower id), written
// in ascending id to ids[0..K) with renormalised softmax weights w[0..K).
// One warp.  L: this warp's shared scratch of E words; ex: K floats.
// Up to 256 logits and K <= 8: merged sorted lists (select_topk_merge), with
// no reduction per pick.  Otherwise, and where that cannot decide the K-th
// pick exactly, a lane keeps the best key of its own logits (ids lane,
// lane+32, ...); each pick is a warp maximum of the lanes' bests (redux),
// then the lowest id holding it, after which only the winning lane rescans
// its own logits.
__device__ inline void select_topk_keys(int E, int K, uint32_t* Lk, float* ex, int* ids, float* w,
                                        int lane);

__device__ inline void select_topk_warp(const float* lg, int E, int K, float* L, float* ex,
                                        int* ids, float* w, int lane) {
    uint32_t* Lk = reinterpret_cast<uint32_t*>(L);
    // the logits come from L2: eight loads in flight a round trip
#pragma unroll 1
    for (int e0 = lane; e0 < E; e0 += 8 * 32) {
        float v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = (e0 + 32 * j < E) ? __ldcg(lg + e0 + 32 * j) : 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (e0 + 32 * j < E) Lk[e0 + 32 * j] = logit_key(v[j]);
    }
    select_topk_keys(E, K, Lk, ex, ids, w, lane);
}

// The softmax weights of a selected set, the same arithmetic whichever way
// the set was found: lane k < K holds pick k (id mye, order-preserving key
// myk), mk is the largest key of the set.  ids ascending, renormalised.
__device__ __forceinline__ void topk_weights(int K, uint32_t myk, uint32_t mye, uint32_t mk,
                                             int rank, float* ex, int* ids, float* w, int lane) {
    float e_k = 0.0f;
    if (lane < K) {
        e_k = expf(key_logit(myk) - key_logit(mk));
        ex[rank] = e_k;
        ids[rank] = int(mye);
    }
    __syncwarp();
    float sum = 0.0f;
    for (int r = 0; r < K; ++r) sum += ex[r];                 // ascending id
    if (lane < K) w[rank] = e_k / sum;
    __syncwarp();
}

// The selection itself on the order-preserving keys Lk[0..E) already in
// this warp's shared scratch (lane-strided writes).  Each lane copies its
// keys (ids lane, lane + 32, ...) into registers, so after a pick only the
// winning lane rescans, in registers.  KPL: keys a lane, >= E / 32.
template <int KPL>
__device__ inline void select_topk_reg(int E, int K, const uint32_t* Lk, float* ex, int* ids,
                                       float* w, int lane) {
    __syncwarp();
    uint32_t key[KPL];
#pragma unroll
    for (int i = 0; i < KPL; ++i) key[i] = lane + 32 * i < E ? Lk[lane + 32 * i] : 0u;
    uint32_t bk = 0u, be = 0x7fffffffu;          // ascending ids: the first maximum stays
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E && (be == 0x7fffffffu || key[i] > bk)) {
            bk = key[i];
            be = uint32_t(e);
        }
    }
    uint32_t myk = 0u, mye = 0x7fffffffu;
    for (int k = 0; k < K; ++k) {
        const uint32_t kmax = __reduce_max_sync(0xffffffffu, bk);
        const uint32_t emin = __reduce_min_sync(0xffffffffu, bk == kmax ? be : 0x7fffffffu);
        if (lane == k) {
            myk = kmax;
            mye = emin;
        }
        if (emin < uint32_t(E) && int(emin & 31u) == lane) {
            // the pick is taken (key 0 never wins); rescan this lane's keys
            bk = 0u;
            be = 0x7fffffffu;
#pragma unroll
            for (int i = 0; i < KPL; ++i) {
                const int e = lane + 32 * i;
                if (uint32_t(e) == emin) key[i] = 0u;
                if (e < E && (be == 0x7fffffffu || key[i] > bk)) {
                    bk = key[i];
                    be = uint32_t(e);
                }
            }
        }
    }
    const uint32_t mk = __shfl_sync(0xffffffffu, myk, 0);    // the first pick is the largest
    int rank = 0;
    for (int j = 0; j < K; ++j) rank += (__shfl_sync(0xffffffffu, mye, j) < mye) ? 1 : 0;
    topk_weights(K, myk, mye, mk, rank, ex, ids, w, lane);
}

// Eight u32 in registers, descending (a bitonic sorting network).
__device__ __forceinline__ void cas_desc(uint32_t& a, uint32_t& b) {
    const uint32_t hi = max(a, b), lo = min(a, b);
    a = hi;
    b = lo;
}
__device__ __forceinline__ void sort8_desc(uint32_t (&a)[8]) {
#pragma unroll
    for (int k = 2; k <= 8; k <<= 1)
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1)
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int l = i ^ j;
                if (l > i) {
                    if ((i & k) == 0)
                        cas_desc(a[i], a[l]);
                    else
                        cas_desc(a[l], a[i]);
                }
            }
}

// Top-K (K <= 8) of E <= 256 keys without a warp reduction per pick.  A
// logit's sort word is its key with the low 8 bits replaced by 255 - id:
// distinct words, ordered by key and, within equal upper bits, by lower id.
// A lane sorts its eight words; five butterfly rounds merge the lanes'
// lists (the larger halves of a list against its partner's reversed list
// hold the top eight of both, then a bitonic merge sorts them), keeping the
// largest word dropped on the way, so every lane ends with the top eight
// words and the ninth.  The set equals the exact top-K unless the K-th and
// (K+1)-th words agree in their upper 24 bits (keys that close, or NaN keys):
// then the function returns false and the exact selection runs instead.
__device__ inline bool select_topk_merge(int E, int K, const uint32_t* Lk, float* ex, int* ids,
                                         float* w, int lane) {
    __syncwarp();
    uint32_t t[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int e = lane + 32 * i;
        t[i] = e < E ? ((Lk[e] & 0xFFFFFF00u) | uint32_t(255 - e)) : 0u;
    }
    sort8_desc(t);
    uint32_t d9 = 0u;                          // the largest word dropped so far
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        uint32_t b[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) b[i] = __shfl_xor_sync(0xffffffffu, t[i], d);
        uint32_t dm = __shfl_xor_sync(0xffffffffu, d9, d);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            dm = max(dm, min(t[i], b[7 - i]));
            t[i] = max(t[i], b[7 - i]);
        }
        d9 = max(d9, dm);
#pragma unroll
        for (int j = 4; j > 0; j >>= 1)
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if ((i ^ j) > i) cas_desc(t[i], t[i ^ j]);
    }
    uint32_t cK = 0u, nxt = d9, myc = 0u;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (i == K - 1) cK = t[i];
        if (i == K) nxt = t[i];
        if (i == lane) myc = t[i];
    }
    const uint32_t up = cK & 0xFFFFFF00u;
    if (up == 0u || up == (nxt & 0xFFFFFF00u)) return false;     // warp-uniform
    // the largest key of the set: among the words whose upper bits equal the
    // first word's (usually the first alone)
    const uint32_t up0 = t[0] & 0xFFFFFF00u;
    uint32_t mk = Lk[255u - (t[0] & 255u)];
#pragma unroll
    for (int j = 1; j < 8; ++j)
        if (j < K && (t[j] & 0xFFFFFF00u) == up0) mk = max(mk, Lk[255u - (t[j] & 255u)]);
    const uint32_t mye = 255u - (myc & 255u);
    int rank = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j)
        if (j < K && 255u - (t[j] & 255u) < mye) ++rank;
    const uint32_t myk = lane < K ? Lk[mye] : 0u;
    topk_weights(K, myk, mye, mk, rank, ex, ids, w, lane);
    return true;
}

__device__ inline void select_topk_keys(int E, int K, uint32_t* Lk, float* ex, int* ids, float* w,
                                        int lane) {
    if (E <= 256 && K <= 8 && select_topk_merge(E, K, Lk, ex, ids, w, lane)) return;
    if (E <= 32)
        select_topk_reg<1>(E, K, Lk, ex, ids, w, lane);
    else if (E <= 64)
        select_topk_reg<2>(E, K, Lk, ex, ids, w, lane);
    else if (E <= 128)
        select_topk_reg<4>(E, K, Lk, ex, ids, w, lane);
    else if (E <= 256)
        select_topk_reg<8>(E, K, Lk, ex, ids, w, lane);
    else if (E <= 512)
        select_topk_reg<16>(E, K, Lk, ex, ids, w, lane);
    else
        select_topk_reg<32>(E, K, Lk, ex, ids, w, lane);
}

// Routing of all T tokens by one CTA into shared memory: s_ids, s_w [T*K],
// s_sig [T].  forced_ids / forced_w replace the selection when given.
// scratch: (nthr / 32) * (E + 16) floats.
template <typename Sync>
__device__ void route_cta(const float* logits, int T, int E, int K, const int32_t* forced_ids,
                          const float* forced_w, int* s_ids, float* s_w, float* s_sig,
                          float* scratch, uint32_t* err, int tid, int nthr, Sync sync) {
    const int lane = tid & 31, wid = tid >> 5, wpb = nthr >> 5;
    const int ldl = E + 1;
    #pragma unroll 1
    for (int t = wid; t < T; t += wpb) {
        const float* lg = logits + size_t(t) * ldl;
        if (forced_ids) {
            #pragma unroll 1
            for (int k = lane; k < K; k += 32) {
                const int id = __ldg(forced_ids + t * K + k);
                if (id < 0 || id >= E) latch(err, STRATA_EBADROUTE);
                s_ids[t * K + k] = id;
                s_w[t * K + k] = __ldg(forced_w + t * K + k);
            }
            if (lane == 0) s_sig[t] = 1.0f / (1.0f + expf(-__ldcg(lg + E)));
        } else {
            // the gate logit is requested with the others
            const float gl = lane == 0 ? __ldcg(lg + E) : 0.0f;
            float* L = scratch + size_t(wid) * (E + 16);
            select_topk_warp(lg, E, K, L, L + E, s_ids + t * K, s_w + t * K, lane);
            if (lane == 0) s_sig[t] = 1.0f / (1.0f + expf(-gl));
        }
    }
    sync();
}

// ---------------------------------------------------------- x activations
// Lane `lane` owns chunks c = lane + 32 m (m < MC) of a length-H row; a chunk
// is 32 elements.  Loads token row x (bf16) as fp32 pairs plus chunk sums.
template <int MC>
__device__ __forceinline__ void load_x(const uint16_t* xrow, int NC, int lane,
                                       uint64_t (&x2)[MC][16], float (&X)[MC]) {
#pragma unroll
    for (int m = 0; m < MC; ++m) {
        const int c = lane + 32 * m;
        float sum = 0.0f;
        if (c < NC) {
            const uint4* p = reinterpret_cast<const uint4*>(xrow + 32 * c);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const uint4 u = ldg_keep(p + v);
                const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float lo = bf16_lo(wv[i]), hi = bf16_hi(wv[i]);
                    x2[m][4 * v + i] = pk(lo, hi);
                    sum += lo + hi;
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) x2[m][j] = 0ull;
        }
        X[m] = sum;
    }
}

// The same from shared memory: a token's row stored chunk-interleaved, the
// 16-byte piece v of chunk c at piece index v * NC + c, so the 32 lanes of a
// warp read 32 consecutive pieces.  Same values and sums as load_x.
template <int MC>
__device__ __forceinline__ void load_x_smem(const uint4* xs, int NC, int lane,
                                            uint64_t (&x2)[MC][16], float (&X)[MC]) {
#pragma unroll
    for (int m = 0; m < MC; ++m) {
        const int c = lane + 32 * m;
        float sum = 0.0f;
        if (c < NC) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const uint4 u = xs[v * NC + c];
                const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float lo = bf16_lo(wv[i]), hi = bf16_hi(wv[i]);
                    x2[m][4 * v + i] = pk(lo, hi);
                    sum += lo + hi;
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) x2[m][j] = 0ull;
        }
        X[m] = sum;
    }
}

}  // namespace strata
