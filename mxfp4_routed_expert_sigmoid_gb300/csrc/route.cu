// Router and token -> expert permutation.
//
// Router (llama.cpp PR #26185 "model: add Kimi-K3 text model", review by
// GrEarl, section "Dry run": 896 experts, 16 used, sigmoid expert-score
// gating, exp_probs_b selection bias):
//   l = <x, W_r[e]> (bf16 products, fp32 accumulation), s = 1 / (1 + expf(-l)),
//   selection key s + b (fp32), top-k with ties to the lower index, slots in
//   key order, w = s / sum(s) over the selected experts (sum in slot order).
//
// Top-k: one CTA per token, thread e holding the key of expert e as a 64-bit
// integer (order-preserving fp32 bits of s + b in the high word, ~expert in
// the low word, so the larger key wins and equal scores fall to the lower
// index).  The k-th largest of the warp maxima bounds the selection from
// below; the few keys above it are ranked by counting (bisection on
// block-wide counts when too many qualify).  Keys are unique, so the result
// is deterministic.
//
// Permutation: histogram of the selection, exclusive scan, and a stable
// scatter that lists each expert's pairs in ascending token order, plus the
// inverse map and the ascending list of experts that received any token
// (small selections: one block sort of (expert, pair) keys).
#include <algorithm>
#include <mutex>

#include "common.cuh"

namespace k3 {
namespace {

constexpr int kMaxE = 1024;   // experts handled by the one-key-per-thread top-k

__device__ __forceinline__ uint32_t order_bits(float v) {
    uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float sigmoid_f32(float l) { return 1.0f / (1.0f + expf(-l)); }

__device__ __forceinline__ uint64_t expert_key(float l, float b, int e) {
    // order-preserving bits of s + b in the high word, ~e in the low word: the
    // larger key is the larger score, and equal scores go to the lower index
    return (static_cast<uint64_t>(order_bits(sigmoid_f32(l) + b)) << 32) |
           static_cast<uint32_t>(0xFFFFFFFFu - static_cast<uint32_t>(e));
}

constexpr int kCand = 64;  // candidate keys ranked by counting

// The top-k of one token by one CTA of kMaxE threads, thread e holding the
// key of expert e (0 for e >= E).  Exactly k keys are chosen (keys are
// unique), listed in key order: idx / w (w = s / sum(s), the sum in slot
// order) are written unless `dry`; returns whether this thread's expert was
// chosen.
//
// Fast path: the k-th largest of the 32 warp maxima, M, bounds the selection
// from below (the k warps whose maxima are >= M hold k distinct keys >= M), so
// the chosen keys are among those >= M.  When at most kCand keys qualify they
// are ranked by counting.  Otherwise (equal or clustered scores) the k-th
// largest high word is found by bisection on its bits with block-wide counts;
// if more experts share it than are still needed, a second bisection on the
// low words keeps the lower experts, and the chosen keys are ranked by
// counting.  Both paths choose the same k keys.  Kept out of line so that a dry
// run (before the logits exist) brings its code into the instruction cache
// ahead of the real one.
__device__ __noinline__ bool select_topk(uint64_t key, float s, int k, int32_t* idx_out, float* w_out,
                                         bool dry) {
    __shared__ uint64_t wmax_s[kMaxE / 32];
    __shared__ uint64_t cand_key[kCand];
    __shared__ float cand_s[kCand];
    __shared__ uint64_t thr_s;
    __shared__ int ncand_s;
    __shared__ uint32_t chosen_bits[kMaxE / 32];
    __shared__ float chosen_s[32];
    constexpr uint32_t kFull = 0xffffffffu;
    const int e = threadIdx.x, lane = e & 31, wid = e >> 5;
    const uint32_t lanes_below = (1u << lane) - 1u;
    uint64_t m = key;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const uint64_t v = __shfl_xor_sync(kFull, m, o);
        m = v > m ? v : m;
    }
    if (lane == 0) wmax_s[wid] = m;
    if (e == 0) ncand_s = 0;
    __syncthreads();
    if (wid == 0) {
        const uint64_t mine = wmax_s[lane];
        int r = 0;
#pragma unroll 8
        for (int j = 0; j < kMaxE / 32; ++j) r += wmax_s[j] > mine ? 1 : 0;
        // the k-th largest maximum; 0 (no bound) when fewer than k warps hold experts
        const uint32_t at = __ballot_sync(kFull, r == k - 1);
        const uint64_t M = at ? __shfl_sync(kFull, mine, __ffs(at) - 1) : 0;
        if (lane == 0) thr_s = M;
    }
    __syncthreads();
    const uint64_t M = thr_s;
    const bool cand = M != 0 && key >= M;
    const uint32_t cbal = __ballot_sync(kFull, cand);
    int base = 0;
    if (lane == 0 && cbal) base = atomicAdd(&ncand_s, __popc(cbal));
    base = __shfl_sync(kFull, base, 0);
    if (cand) {
        const int pos = base + __popc(cbal & lanes_below);
        if (pos < kCand) {
            cand_key[pos] = key;
            cand_s[pos] = s;
        }
    }
    __syncthreads();
    const int n = ncand_s;
    if (M != 0 && n <= kCand) {
        if (e < 32) chosen_bits[e] = 0;
        __syncthreads();
        if (e < n) {
            const uint64_t kk = cand_key[e];
            int rank = 0;
            for (int j = 0; j < n; ++j) rank += cand_key[j] > kk ? 1 : 0;
            if (rank < k) {
                const int ex = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(kk));
                chosen_s[rank] = cand_s[e];
                if (!dry) idx_out[rank] = ex;
                atomicOr(&chosen_bits[ex >> 5], 1u << (ex & 31));
            }
        }
    } else {
        const uint32_t hi = static_cast<uint32_t>(key >> 32), lo = static_cast<uint32_t>(key);
        uint32_t H = 0;
        for (int bit = 31; bit >= 0; --bit) {
            const uint32_t c = H | (1u << bit);
            if (__syncthreads_count(hi >= c) >= k) H = c;
        }
        const int need = k - __syncthreads_count(hi > H);
        uint32_t L = 0;
        if (__syncthreads_count(hi == H) > need) {
            for (int bit = 31; bit >= 0; --bit) {
                const uint32_t c = L | (1u << bit);
                if (__syncthreads_count(hi == H && lo >= c) >= need) L = c;
            }
        }
        const bool chosen = key != 0 && (hi > H || (hi == H && lo >= L));
        const uint32_t bal = __ballot_sync(kFull, chosen);
        if (lane == 0) chosen_bits[wid] = bal;
        __syncthreads();
        if (chosen) {
            int pos = __popc(bal & lanes_below);
            for (int w = 0; w < wid; ++w) pos += __popc(chosen_bits[w]);
            cand_key[pos] = key;
        }
        __syncthreads();
        if (chosen) {
            int rank = 0;
            for (int j = 0; j < k; ++j) rank += cand_key[j] > key ? 1 : 0;
            chosen_s[rank] = s;
            if (!dry) idx_out[rank] = e;
        }
    }
    __syncthreads();
    if (e < k) {
        float sum = 0.0f;
        for (int j = 0; j < k; ++j) sum += chosen_s[j];
        if (!dry) w_out[e] = chosen_s[e] / sum;
    }
    const bool mine = (chosen_bits[wid] >> lane) & 1u;
    __syncthreads();
    return mine;
}

// Top-k and weights of token blockIdx.x (blockDim.x == kMaxE).  With
// a.active set (decode), the ascending list of experts that received any token
// (count at active[E]) is written too: by the CTA itself for one token;
// otherwise every chosen expert is marked in the bitmap kept in the workspace
// header, and the last CTA turns the bitmap into the list and clears it.  The bias is read and the selection rehearsed on it before the
// logits are awaited, so both overlap the logits kernel.
__global__ void __launch_bounds__(kMaxE)
route_topk_kernel(RouteArgs a) {
    __shared__ uint32_t ticket_s;
    const int t = blockIdx.x, e = threadIdx.x, lane = e & 31;
    const bool valid = e < a.E;
    const float b = valid ? a.bias[e] : 0.0f;
    select_topk(valid ? expert_key(0.0f, b, e) : 0, 0.5f, a.k, nullptr, nullptr, true);
    pdl_wait();
    pdl_trigger();
    StampScope stamp(a.st_b);
    const float l = valid ? a.logits[static_cast<size_t>(t) * a.E + e] : 0.0f;
    // a logit that is not finite, or a NaN bias (a bias of +-inf orders like
    // any other key), leaves the selection undefined: flagged
    if (__syncthreads_or(valid && (!isfinite(l) || isnan(b))) && e == 0) set_error(a.hdr, K3MOE_ERR_NONFINITE, 1);
    const bool chosen = select_topk(valid ? expert_key(l, b, e) : 0, sigmoid_f32(l), a.k,
                                    a.idx + static_cast<size_t>(t) * a.k,
                                    a.wts + static_cast<size_t>(t) * a.k, false);
    if (!a.active) return;
    if (gridDim.x == 1) {
        // one token: its selection, in ascending expert order, is the active
        // list (warp w's chosen experts start at the prefix of the warp counts)
        __shared__ int wbase[kMaxE / 32 + 1];
        const uint32_t bal = __ballot_sync(0xffffffffu, chosen);
        if (lane == 0) wbase[e >> 5] = __popc(bal);
        __syncthreads();
        if (e < 32) {
            const int c = wbase[lane];
            int incl = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            __syncwarp();
            wbase[lane] = incl - c;
            if (lane == 31) wbase[32] = incl;
        }
        __syncthreads();
        if (chosen) a.active[wbase[e >> 5] + __popc(bal & ((1u << lane) - 1u))] = e;
        if (e == 0) a.active[a.E] = wbase[32];
        return;
    }
    if (chosen) atomicOr(&a.hdr->pad[e >> 5], 1u << (e & 31));
    __threadfence();
    __syncthreads();
    if (e == 0) ticket_s = atomicAdd(&a.hdr->counters[CTR_ROUTE], 1u);
    __syncthreads();
    if (ticket_s != gridDim.x - 1 || e >= 32) return;
    __threadfence();
    volatile uint32_t* bitmap = a.hdr->pad;
    const uint32_t word = bitmap[lane];
    const int c = __popc(word);
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    int pos = incl - c;
    for (uint32_t w = word; w != 0; w &= w - 1) a.active[pos++] = 32 * lane + (__ffs(w) - 1);
    if (lane == 31) a.active[a.E] = incl;
    bitmap[lane] = 0;
    if (lane == 0) a.hdr->counters[CTR_ROUTE] = 0;
}

// Top-k of many tokens (the permutation path, no active list), one warp per
// token: lane l holds the keys of experts l, l + 32, ... (up to 32 each) in
// registers.  The k-th largest of the 32 lane maxima, M, bounds the selection
// from below (the k lanes whose maxima are >= M hold k keys >= M), so the
// chosen keys are among those >= M; when at most kCandW of them qualify they
// are gathered in shared memory and ranked by counting.  Otherwise k rounds
// each take the warp's largest remaining key (a butterfly maximum over the
// lanes' own maxima).  Keys are unique, so either way the slots come out in
// key order exactly as in the one-CTA-per-token kernel, and the weights are
// formed the same way (w = s / sum(s), the sum in slot order): the result is
// bitwise that kernel's.
constexpr int kTopkWarpTokens = 8;   // tokens (warps) per CTA
constexpr int kTopkWarpMinT = 2048;  // up to this many tokens: one block per token
constexpr int kCandW = 64;           // candidates ranked by counting
__global__ void __launch_bounds__(32 * kTopkWarpTokens)
route_topk_warp_kernel(RouteArgs a) {
    __shared__ uint64_t cand_s[kTopkWarpTokens][kCandW];
    __shared__ int slot_s[kTopkWarpTokens][32];
    pdl_wait();
    pdl_trigger();
    StampScope stamp(a.st_b);
    constexpr uint32_t kFull = 0xffffffffu;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int t = blockIdx.x * kTopkWarpTokens + wid;
    if (t >= a.T) return;
    const float* lrow = a.logits + static_cast<size_t>(t) * a.E;
    uint64_t key[kMaxE / 32];
    bool bad = false;
#pragma unroll
    for (int j = 0; j < kMaxE / 32; ++j) {
        const int e = lane + 32 * j;
        key[j] = 0;
        if (e < a.E) {
            const float l = lrow[e], b = a.bias[e];
            bad |= !isfinite(l) || isnan(b);
            key[j] = expert_key(l, b, e);
        }
    }
    // a logit that is not finite, or a NaN bias, leaves the selection undefined: flagged
    if (__any_sync(kFull, bad) && lane == 0) set_error(a.hdr, K3MOE_ERR_NONFINITE, 1);
    uint64_t mine = 0;
#pragma unroll
    for (int j = 0; j < kMaxE / 32; ++j) mine = key[j] > mine ? key[j] : mine;
    // rank of this lane's maximum among the lane maxima; M = the one ranked k - 1
    int rk = 0;
    for (int o = 1; o < 32; ++o) rk += __shfl_sync(kFull, mine, (lane + o) & 31) > mine ? 1 : 0;
    const uint32_t at = __ballot_sync(kFull, rk == a.k - 1 && mine != 0);
    const uint64_t M = at ? __shfl_sync(kFull, mine, __ffs(at) - 1) : 0;
    int cnt = 0;
#pragma unroll
    for (int j = 0; j < kMaxE / 32; ++j) cnt += (M != 0 && key[j] >= M) ? 1 : 0;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += v;
    }
    const int n = __shfl_sync(kFull, incl, 31);
    if (M != 0 && n <= kCandW) {
        int pos = incl - cnt;
#pragma unroll
        for (int j = 0; j < kMaxE / 32; ++j)
            if (key[j] >= M) cand_s[wid][pos++] = key[j];
        __syncwarp();
        for (int c = lane; c < n; c += 32) {
            const uint64_t kc = cand_s[wid][c];
            int r = 0;
            for (int q = 0; q < n; ++q) r += cand_s[wid][q] > kc ? 1 : 0;
            if (r < a.k) slot_s[wid][r] = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(kc));
        }
    } else {
        for (int r = 0; r < a.k; ++r) {
            uint64_t m = mine;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const uint64_t v = __shfl_xor_sync(kFull, m, o);
                m = v > m ? v : m;
            }
            if (mine == m) {  // this lane holds the round's key: drop it
                uint64_t nm = 0;
#pragma unroll
                for (int j = 0; j < kMaxE / 32; ++j) {
                    if (key[j] == m) key[j] = 0;
                    nm = key[j] > nm ? key[j] : nm;
                }
                mine = nm;
            }
            if (lane == 0) slot_s[wid][r] = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(m));
        }
    }
    __syncwarp();
    const int slot_e = lane < a.k ? slot_s[wid][lane] : 0;  // lane r < k: the expert of slot r
    const float sj = lane < a.k ? sigmoid_f32(lrow[slot_e]) : 0.0f;
    float sum = 0.0f;
    for (int j = 0; j < a.k; ++j) sum += __shfl_sync(kFull, sj, j);
    if (lane < a.k) {
        a.idx[static_cast<size_t>(t) * a.k + lane] = slot_e;
        a.wts[static_cast<size_t>(t) * a.k + lane] = sj / sum;
    }
}

// exclusive scan of n <= 4 * blockDim ints in shared memory (in place);
// returns the total.  Requires blockDim.x == 256.
__device__ int block_exclusive_scan(int* data, int n) {
    __shared__ int warp_tot[8];
    __shared__ int total_s;
    const int tid = threadIdx.x;
    int v[4];
    int local = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int p = tid * 4 + i;
        v[i] = p < n ? data[p] : 0;
        local += v[i];
    }
    // inclusive warp scan of the per-thread totals
    int incl = local;
    const int lane = tid & 31, wid = tid >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) warp_tot[wid] = incl;
    __syncthreads();
    if (tid == 0) {
        int run = 0;
        for (int w = 0; w < 8; ++w) {
            int t = warp_tot[w];
            warp_tot[w] = run;
            run += t;
        }
        total_s = run;
    }
    __syncthreads();
    int run = warp_tot[wid] + incl - local;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int p = tid * 4 + i;
        if (p < n) data[p] = run;
        run += v[i];
    }
    __syncthreads();
    return total_s;
}

// Logits by GEMV (one warp per expert at T = 1, two per expert for more
// tokens, all T tokens).  Each warp issues all loads of its part of the
// weight row before it needs them; the T token rows are staged once per CTA
// in shared memory.  With xq requested, CTAs past those that compute logits
// write the token rows as E2M1 terms for the expert kernels, one warp per
// 32-element block.
constexpr int kRouteChunks = 16;  // 16-byte weight loads per lane in flight

// One warp's logits of expert e: lane l holds the weight elements 256 i +
// 8 l .. 256 i + 8 l + 7 (wv, loaded by the caller; rows longer than 256
// kRouteChunks are fetched here in further rounds) and multiplies them with
// the token rows staged in xs; a token's products add in the order chunk,
// q = 0..3, low half before high half.  gemv_part_tokens takes up to eight
// tokens over part of a row, one token's chunk after the other; gemv_row_one
// is the whole row for a single token without the per-token guards (it
// measured 3.7 against 4.2 us for the whole router at T = 1).
template <typename Body>
__device__ __forceinline__ void gemv_chunks(int k0, int k1, int lane, const uint16_t* wrow,
                                            uint4 (&wv)[kRouteChunks], Body body) {
    for (int base = k0; base < k1; base += 256 * kRouteChunks) {
        if (base > k0) {
#pragma unroll
            for (int i = 0; i < kRouteChunks; ++i) {
                const int c = base + i * 256 + lane * 8;
                wv[i] = c < k1 ? ldg_nc_v4(wrow + c) : make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int i = 0; i < kRouteChunks; ++i) {
            const int c = base + i * 256 + lane * 8;
            if (c >= k1) break;
            body(wv[i], c);
        }
    }
}

__device__ __forceinline__ float dot8_bf16(const uint4& w, const uint4& x, float acc) {
    const uint32_t wq[4] = {w.x, w.y, w.z, w.w}, xq[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        acc = fmaf(__uint_as_float(wq[q] << 16), __uint_as_float(xq[q] << 16), acc);
        acc = fmaf(__uint_as_float(wq[q] & 0xFFFF0000u), __uint_as_float(xq[q] & 0xFFFF0000u), acc);
    }
    return acc;
}

__device__ __forceinline__ void gemv_row_one(const RouteArgs& a, int e, int lane, const uint16_t* wrow,
                                             uint4 (&wv)[kRouteChunks], const uint4* xs) {
    float acc = 0.0f;
    gemv_chunks(0, a.d_r, lane, wrow, wv, [&](const uint4& w, int c) { acc = dot8_bf16(w, xs[c / 8], acc); });
    const float v = warp_sum(acc);
    if (lane == 0) a.logits[e] = v;
}

// Up to eight tokens over inputs [k0, k1) of a row, one token's chunk after
// the other: the warp's per-token sums go to part[0 .. T) (lane 0 writes).
__device__ __forceinline__ void gemv_part_tokens(const RouteArgs& a, int k0, int k1, int lane,
                                                 const uint16_t* wrow, uint4 (&wv)[kRouteChunks],
                                                 const uint4* xs, float* part) {
    float acc[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) acc[t] = 0.0f;
    gemv_chunks(k0, k1, lane, wrow, wv, [&](const uint4& w, int c) {
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            if (t >= a.T) break;
            acc[t] = dot8_bf16(w, xs[(t * a.d_r + c) / 8], acc[t]);
        }
    });
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        if (t >= a.T) break;
        const float v = warp_sum(acc[t]);
        if (lane == 0) part[t] = v;
    }
}

// Rows per logits CTA: one warp per row for one token; for more tokens two
// warps per row, each multiplying half of the row's 256-wide chunks, so that
// a warp's chains are half as long (the two halves' sums are then added,
// half 0 first).
__host__ __device__ inline int route_rows_per_cta(int T) { return T == 1 ? 8 : 4; }

__global__ void __launch_bounds__(256)
route_small_kernel(RouteArgs a) {
    extern __shared__ __align__(16) uint4 xs[];  // [T * d_r / 8]
    // the top-k kernel may start launching now: it waits for this grid's
    // completion (griddepcontrol.wait) before reading the logits
    pdl_trigger();
    StampScope stamp(a.st_a);
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int rpc = route_rows_per_cta(a.T);
    const int gemv_ctas = (a.E + rpc - 1) / rpc;
    if (static_cast<int>(blockIdx.x) >= gemv_ctas) {
        const int nb = a.d_r / 32;
        const int xq_ctas = gridDim.x - gemv_ctas;
        for (int i = (blockIdx.x - gemv_ctas) * 8 + wid; i < a.T * nb; i += xq_ctas * 8) {
            const int t = i / nb, b = i - t * nb;
            uint32_t q[kTerms], sb[kTerms];
            quantize_terms(bf16_to_f32(a.x[static_cast<size_t>(t) * a.d_r + 32 * b + lane]), q, sb);
            store_terms(q, sb, t, b & 7, a.xq + static_cast<size_t>(b >> 3) * a.xq_n * 128,
                        a.xsf + static_cast<size_t>(b >> 3) * 1024);
        }
        return;
    }
    // this warp's row and inputs [k0, k1) of it
    const int half = rpc == 8 ? 0 : (wid & 1);
    const int e = blockIdx.x * rpc + (rpc == 8 ? wid : wid >> 1);
    const int nch = (a.d_r + 255) / 256, hch = rpc == 8 ? nch : (nch + 1) / 2;
    const int k0 = half * hch * 256, k1 = min(a.d_r, (half + 1) * hch * 256);
    const uint16_t* wrow = a.w + static_cast<size_t>(e < a.E ? e : 0) * a.d_r;
    uint4 wv[kRouteChunks];
#pragma unroll
    for (int i = 0; i < kRouteChunks; ++i) {
        const int c = k0 + i * 256 + lane * 8;
        wv[i] = (e < a.E && c < k1) ? ldg_nc_v4(wrow + c) : make_uint4(0, 0, 0, 0);
    }
    // the token rows into shared memory, eight loads per thread in flight
    // before their stores (T = 8 rows of 3584 are 14 loads per thread)
    const int nvec = a.T * a.d_r / 8;
    constexpr int kStageLoads = 8;
    for (int v0 = threadIdx.x; v0 < nvec; v0 += kStageLoads * blockDim.x) {
        uint4 xv[kStageLoads];
#pragma unroll
        for (int j = 0; j < kStageLoads; ++j) {
            const int v = v0 + j * blockDim.x;
            if (v < nvec) xv[j] = reinterpret_cast<const uint4*>(a.x)[v];
        }
#pragma unroll
        for (int j = 0; j < kStageLoads; ++j) {
            const int v = v0 + j * blockDim.x;
            if (v < nvec) xs[v] = xv[j];
        }
    }
    __syncthreads();

    if (a.T == 1) {
        if (e < a.E) gemv_row_one(a, e, lane, wrow, wv, xs);
        return;
    }
    __shared__ float part_s[8][8];  // [warp][token]
    if (e < a.E) gemv_part_tokens(a, k0, k1, lane, wrow, wv, xs, part_s[wid]);
    __syncthreads();
    if (half == 0 && e < a.E && lane < a.T)
        a.logits[static_cast<size_t>(lane) * a.E + e] = part_s[wid][lane] + part_s[wid + 1][lane];
}

// Plain tiled SIMT logits for moderate T: 64 tokens x 64 experts per CTA.
__global__ void __launch_bounds__(256)
logits_simt_kernel(RouteArgs a) {
    StampScope stamp(a.st_a);
    __shared__ float xs[64][33];
    __shared__ float ws[64][33];
    const int t0 = blockIdx.y * 64, e0 = blockIdx.x * 64;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;  // 16 x 16 threads, 4x4 each
    float acc[4][4] = {};
    for (int c0 = 0; c0 < a.d_r; c0 += 32) {
        for (int i = threadIdx.x; i < 64 * 32; i += 256) {
            const int r = i >> 5, c = i & 31;
            const int t = t0 + r, e = e0 + r;
            xs[r][c] = (t < a.T) ? bf16_to_f32(a.x[static_cast<size_t>(t) * a.d_r + c0 + c]) : 0.0f;
            ws[r][c] = (e < a.E) ? bf16_to_f32(a.w[static_cast<size_t>(e) * a.d_r + c0 + c]) : 0.0f;
        }
        __syncthreads();
#pragma unroll 8
        for (int c = 0; c < 32; ++c) {
            float xv[4], wv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                xv[i] = xs[ty * 4 + i][c];
                wv[i] = ws[tx * 4 + i][c];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xv[i], wv[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int t = t0 + ty * 4 + i, e = e0 + tx * 4 + j;
            if (t < a.T && e < a.E) a.logits[static_cast<size_t>(t) * a.E + e] = acc[i][j];
        }
}

// ---- chunked permutation for any T ----------------------------------------
constexpr int kChunk = 64;  // tokens per chunk

__global__ void __launch_bounds__(256)
perm_count_kernel(int32_t* __restrict__ idx, int T, int k, int E, int32_t* chunk_cnt, WsHeader* hdr,
                  int clamp, uint64_t* st) {
    StampScope stamp(st);
    extern __shared__ int hist[];
    const int c = blockIdx.x;
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    const int t0 = c * kChunk, t1 = min(T, t0 + kChunk);
    for (int p = t0 * k + threadIdx.x; p < t1 * k; p += blockDim.x) {
        int e = idx[p];
        if (e < 0 || e >= E) {
            // an expert outside [0, E): recorded; with clamp (a selection copied into
            // the workspace) the entry becomes expert 0, so every later index stays in range
            set_error(hdr, K3MOE_ERR_INVALID_ARG, 2);
            if (!clamp) continue;
            e = 0;
            idx[p] = 0;
        }
        atomicAdd(&hist[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        chunk_cnt[static_cast<size_t>(c) * E + e] = hist[e];
}

// one CTA: per-expert running sums over chunks, exclusive scan over experts,
// active list
__global__ void __launch_bounds__(256)
perm_scan_kernel(int32_t* chunk_cnt, int nchunks, int E, int P, int32_t* counts,
                 int32_t* offsets, int32_t* active, uint64_t* st) {
    StampScope stamp(st);
    extern __shared__ int sm[];  // [2 * E]
    int* tot = sm;
    int* flag = sm + E;
    // each thread scans the chunk counts of its (at most four) experts, the
    // loads of 16 chunks x 4 experts issued together
    constexpr int kBatch = 16;
    int run[4] = {0, 0, 0, 0};
    for (int c0 = 0; c0 < nchunks; c0 += kBatch) {
        int v[4][kBatch];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int e = threadIdx.x + q * blockDim.x;
#pragma unroll
            for (int i = 0; i < kBatch; ++i)
                v[q][i] = (e < E && c0 + i < nchunks) ? chunk_cnt[static_cast<size_t>(c0 + i) * E + e] : 0;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int e = threadIdx.x + q * blockDim.x;
#pragma unroll
            for (int i = 0; i < kBatch; ++i) {
                if (e < E && c0 + i < nchunks) {
                    chunk_cnt[static_cast<size_t>(c0 + i) * E + e] = run[q];  // exclusive within the expert
                    run[q] += v[q][i];
                }
            }
        }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int e = threadIdx.x + q * blockDim.x;
        if (e < E) {
            tot[e] = run[q];
            counts[e] = run[q];
            flag[e] = run[q] > 0 ? 1 : 0;
        }
    }
    __syncthreads();
    // scan in chunks of 1024 (block_exclusive_scan handles up to 1024 entries)
    int base = 0, abase = 0;
    for (int e0 = 0; e0 < E; e0 += 1024) {
        const int n = min(1024, E - e0);
        const int t = block_exclusive_scan(tot + e0, n);
        const int ta = block_exclusive_scan(flag + e0, n);
        for (int e = threadIdx.x; e < n; e += blockDim.x) {
            offsets[e0 + e] = base + tot[e0 + e];
            if (counts[e0 + e] > 0) active[abase + flag[e0 + e]] = e0 + e;
        }
        base += t;
        abase += ta;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        offsets[E] = P;
        active[E] = abase;
    }
}

// one warp per chunk: tokens in order, slots in parallel (distinct experts)
__global__ void __launch_bounds__(32)
perm_scatter_kernel(const int32_t* __restrict__ idx, int T, int k, int E,
                    const int32_t* __restrict__ chunk_base, const int32_t* __restrict__ offsets,
                    int32_t* perm, int32_t* inv, uint64_t* st) {
    StampScope stamp(st);
    extern __shared__ int running[];
    const int c = blockIdx.x, lane = threadIdx.x;
    for (int e = lane; e < E; e += 32)
        running[e] = offsets[e] + chunk_base[static_cast<size_t>(c) * E + e];
    __syncwarp();
    const int t0 = c * kChunk, t1 = min(T, t0 + kChunk);
    for (int t = t0; t < t1; ++t) {
        if (lane < k) {
            const int p = t * k + lane;
            const int e = idx[p];
            if (e >= 0 && e < E) {
                const int row = running[e];
                running[e] = row + 1;
                perm[row] = p;
                inv[p] = row;
            }
        }
        __syncwarp();
    }
}

}  // namespace

cudaError_t launch_route_topk(const RouteArgs& a_in, cudaStream_t s) {
    RouteArgs a = a_in;
    a.st_b = trace_stamp("route_topk");
    const cudaError_t e = launch_pdl(route_topk_kernel, dim3(a.T), dim3(kMaxE), 0, s, a);
    trace_mark("route_topk", s);
    return e;
}

cudaError_t launch_route_small(const RouteArgs& a_in, cudaStream_t s) {
    RouteArgs a = a_in;
    a.st_a = trace_stamp("route_small");
    const int rpc = route_rows_per_cta(a.T);
    const int gemv_ctas = (a.E + rpc - 1) / rpc;
    const int xq_ctas = a.xq ? std::min(128, (a.T * (a.d_r / 32) + 7) / 8) : 0;
    const size_t smem = static_cast<size_t>(a.T) * a.d_r * 2;
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(route_small_kernel,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    route_small_kernel<<<gemv_ctas + xq_ctas, 256, smem, s>>>(a);
    trace_mark("route_small", s);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_route_topk(a, s);
}

// ---------------------------------------------------------------------------
// Router with library-owned scratch (k3moe_route_noalloc).
//
// The small-T router needs a workspace header (its status word) and, when the
// caller does not want the logits, a [T, E] fp32 buffer for them.  This
// variant keeps both in one file-scope device array instead of a caller
// workspace: it is part of the module image, so every GPU that loads the
// library holds these bytes until the process exits, and every call shares
// them.
// ---------------------------------------------------------------------------
constexpr size_t kNoAllocScratch =
    sizeof(WsHeader) + static_cast<size_t>(kNoAllocMaxT) * kNoAllocMaxE * sizeof(float);
static __device__ __align__(256) unsigned char g_route_scratch[kNoAllocScratch];

// Device address of g_route_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up
// once per device (with that device current) and cached.
static cudaError_t route_scratch_address(void** out) {
    static std::mutex mu;
    static void* addr[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_route_scratch);
        if (e != cudaSuccess) return e;
        addr[dev] = p;
    }
    *out = addr[dev];
    return cudaSuccess;
}

cudaError_t launch_route_noalloc(RouteArgs a, cudaStream_t s) {
    void* scratch = nullptr;
    cudaError_t e = route_scratch_address(&scratch);
    if (e != cudaSuccess) return e;
    // the header (completion counter, status) must start at zero: clear it on
    // the caller's stream, so it is ordered after any earlier call there
    e = cudaMemsetAsync(scratch, 0, sizeof(WsHeader), s);
    if (e != cudaSuccess) return e;
    a.hdr = static_cast<WsHeader*>(scratch);
    if (!a.logits) a.logits = reinterpret_cast<float*>(static_cast<char*>(scratch) + sizeof(WsHeader));
    a.active = nullptr;
    return launch_route_small(a, s);
}

cudaError_t launch_topk(const RouteArgs& a_in, cudaStream_t s) {
    RouteArgs a = a_in;
    a.active = nullptr;  // the permutation kernels list the active experts
    // a block per token finishes a token sooner (9 us for 512 tokens against
    // 15 us with warps), warps cover more tokens at once (58 us for 8192
    // tokens against 150 us with blocks)
    if (a.T <= kTopkWarpMinT) return launch_route_topk(a, s);
    a.st_b = trace_stamp("route_topk");
    const cudaError_t e = launch_pdl(route_topk_warp_kernel, dim3((a.T + kTopkWarpTokens - 1) / kTopkWarpTokens),
                                     dim3(32 * kTopkWarpTokens), 0, s, a);
    trace_mark("route_topk", s);
    return e;
}

cudaError_t launch_logits_simt(const RouteArgs& a_in, cudaStream_t s) {
    RouteArgs a = a_in;
    a.st_a = trace_stamp("logits_simt");
    dim3 grid((a.E + 63) / 64, (a.T + 63) / 64);
    logits_simt_kernel<<<grid, 256, 0, s>>>(a);
    trace_mark("logits_simt", s);
    return cudaGetLastError();
}

size_t permute_scratch_bytes(int T, int E) {
    const size_t nchunks = (static_cast<size_t>(T) + kChunk - 1) / kChunk;
    return align_up(nchunks * E * sizeof(int32_t));
}

cudaError_t launch_permute(const int32_t* idx, int T, int k, int E, int32_t* counts,
                           int32_t* offsets, int32_t* perm, int32_t* inv, int32_t* active,
                           void* scratch, WsHeader* hdr, cudaStream_t s, int clamp) {
    const int nchunks = (T + kChunk - 1) / kChunk;
    int32_t* chunk = static_cast<int32_t*>(scratch);
    const size_t smem = static_cast<size_t>(E) * sizeof(int);
    if (smem > 48 * 1024) {
        cudaFuncSetAttribute(perm_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
        cudaFuncSetAttribute(perm_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    }
    if (2 * smem > 48 * 1024)
        cudaFuncSetAttribute(perm_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(2 * smem));
    perm_count_kernel<<<nchunks, 256, smem, s>>>(const_cast<int32_t*>(idx), T, k, E, chunk, hdr, clamp,
                                                 trace_stamp("perm_count"));
    trace_mark("perm_count", s);
    perm_scan_kernel<<<1, 256, 2 * smem, s>>>(chunk, nchunks, E, T * k, counts, offsets, active,
                                              trace_stamp("perm_scan"));
    trace_mark("perm_scan", s);
    perm_scatter_kernel<<<nchunks, 32, smem, s>>>(idx, T, k, E, chunk, offsets, perm, inv,
                                                  trace_stamp("perm_scatter"));
    trace_mark("perm_scatter", s);
    return cudaGetLastError();
}

}  // namespace k3
