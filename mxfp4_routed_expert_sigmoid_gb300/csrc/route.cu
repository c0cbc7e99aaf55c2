// Router and token -> expert permutation.
//
// Router (llama.cpp PR #26185 "model: add Kimi-K3 text model", review by
// GrEarl, section "Dry run": 896 experts, 16 used, sigmoid expert-score
// gating, exp_probs_b selection bias):
//   l = <x, W_r[e]> (bf16 products, fp32 accumulation), s = 1 / (1 + expf(-l)),
//   selection key s + b (fp32), top-k with ties to the lower index, slots in
//   key order, w = s / sum(s) over the selected experts (sum in slot order).
//
// Top-k: each warp owns one token; every lane holds the keys of experts
// lane, lane+32, ... as 64-bit integers (order-preserving fp32 bits of s + b
// in the high word, ~expert in the low word, so the larger key wins and equal
// scores fall to the lower index); k rounds of a warp-wide max extract the
// selection in slot order.  Keys are unique, so the result is deterministic.
//
// Permutation: histogram of the selection, exclusive scan, and a stable
// scatter that lists each expert's pairs in ascending token order, plus the
// inverse map and the ascending list of experts that received any token.
#include <mutex>

#include "common.cuh"

namespace k3 {
namespace {

constexpr int kMaxE = 1024;   // experts handled by the in-register top-k
constexpr int kKeysPerLane = kMaxE / 32;

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

__device__ __forceinline__ int key_expert(uint64_t key) {
    return static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(key & 0xFFFFFFFFu));
}

// The k largest of the (unique) keys held by the warp, KPL per lane: k rounds
// of a warp-wide max; lane j < k returns the j-th largest.
template <int KPL>
__device__ __forceinline__ uint64_t warp_topk(uint64_t (&key)[KPL], int k) {
    const int lane = threadIdx.x & 31;
    uint64_t mine = 0;
    for (int j = 0; j < k; ++j) {
        uint64_t best = 0;
#pragma unroll
        for (int i = 0; i < KPL; ++i) best = key[i] > best ? key[i] : best;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const uint64_t other = __shfl_xor_sync(0xffffffffu, best, o);
            best = other > best ? other : best;
        }
#pragma unroll
        for (int i = 0; i < KPL; ++i)
            if (key[i] == best) key[i] = 0;
        if (lane == j) mine = best;
    }
    return mine;
}

// The k best experts among [e0, e1) of one token's logits (one warp; at most
// 32 * KPL candidates); lane j < k returns the j-th key.
template <int KPL>
__device__ uint64_t topk_slice(const float* lrow, const float* __restrict__ bias, int e0, int e1,
                               int k, WsHeader* hdr) {
    const int lane = threadIdx.x & 31;
    uint64_t key[KPL];
    bool bad = false;
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
        const int e = e0 + lane + 32 * i;
        key[i] = 0;
        if (e < e1) {
            const float l = lrow[e];
            bad |= !isfinite(l);
            key[i] = expert_key(l, bias[e], e);
        }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) set_error(hdr, K3MOE_ERR_NONFINITE, 1);
    return warp_topk<KPL>(key, k);
}

// Writes the selection of one token from its k winning keys (lane j holds the
// j-th): idx, and the weights s / sum(s) summed in slot order.
__device__ void write_selection(uint64_t mine, const float* lrow, int k, int32_t* __restrict__ idx_out,
                                float* __restrict__ w_out, int32_t* sel_smem) {
    const int lane = threadIdx.x & 31;
    const int e = key_expert(mine);
    const float s_mine = lane < k ? sigmoid_f32(lrow[e]) : 0.0f;
    float sum = 0.0f;
    for (int j = 0; j < k; ++j) sum += __shfl_sync(0xffffffffu, s_mine, j);
    if (lane < k) {
        idx_out[lane] = e;
        w_out[lane] = s_mine / sum;
        if (sel_smem) sel_smem[lane] = e;
    }
}

// top-k of one token by one warp over all E experts
__device__ void topk_token(const float* lrow, const float* __restrict__ bias, int E,
                           int k, int32_t* __restrict__ idx_out, float* __restrict__ w_out,
                           int32_t* sel_smem, WsHeader* hdr) {
    const uint64_t mine = topk_slice<kKeysPerLane>(lrow, bias, 0, E, k, hdr);
    write_selection(mine, lrow, k, idx_out, w_out, sel_smem);
}

// top-k of T <= 8 tokens by the 8 warps of a CTA: G = 8 / T' warps per token
// (T' = T rounded up to a power of two) each keep the k best of a slice of the
// experts, then one warp per token merges the G * k candidates.
template <int G>
__device__ void topk_tokens_cta(const RouteArgs& a, int32_t* sel, uint64_t (*cand)[32]) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int t = wid / G, gw = wid % G;
    const int slice = (a.E + G - 1) / G;
    const float* lrow = a.logits + static_cast<size_t>(t) * a.E;
    if (t < a.T) {
        const int e0 = gw * slice, e1 = min(a.E, e0 + slice);
        const uint64_t mine = topk_slice<32 / G>(lrow, a.bias, e0, e1, a.k, a.hdr);
        if (G == 1) {
            write_selection(mine, lrow, a.k, a.idx + static_cast<size_t>(t) * a.k,
                            a.wts + static_cast<size_t>(t) * a.k, sel + t * a.k);
        } else if (lane < a.k) {
            cand[wid][lane] = mine;
        }
    }
    if (G == 1) return;
    __syncthreads();
    if (t < a.T && gw == 0) {
        constexpr int KPL = (G * 32 + 31) / 32;  // G * k <= G * 32 candidates
        uint64_t key[KPL];
#pragma unroll
        for (int i = 0; i < KPL; ++i) {
            const int c = lane + 32 * i;  // candidate c = (warp c / k, rank c % k)
            key[i] = c < G * a.k ? cand[wid + c / a.k][c % a.k] : 0;
        }
        const uint64_t mine = warp_topk<KPL>(key, a.k);
        write_selection(mine, lrow, a.k, a.idx + static_cast<size_t>(t) * a.k,
                        a.wts + static_cast<size_t>(t) * a.k, sel + t * a.k);
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

// permutation of a small selection held in shared memory (T*k <= 256, E <= 1024)
__device__ void permute_small(const int32_t* sel, int T, int k, int E, int32_t* counts,
                              int32_t* offsets, int32_t* perm, int32_t* inv, int32_t* active) {
    __shared__ int cnt[kMaxE];
    __shared__ int off[kMaxE];
    const int tid = threadIdx.x;
    const int P = T * k;
    for (int e = tid; e < E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    for (int p = tid; p < P; p += blockDim.x) atomicAdd(&cnt[sel[p]], 1);
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) off[e] = cnt[e];
    __syncthreads();
    block_exclusive_scan(off, E);
    for (int e = tid; e < E; e += blockDim.x) {
        counts[e] = cnt[e];
        offsets[e] = off[e];
    }
    if (tid == 0) offsets[E] = P;
    for (int p = tid; p < P; p += blockDim.x) {
        const int e = sel[p];
        int rank = 0;
        for (int q = 0; q < p; ++q) rank += (sel[q] == e);
        const int row = off[e] + rank;
        perm[row] = p;
        inv[p] = row;
    }
    __syncthreads();
    // ascending list of experts that received a token
    for (int e = tid; e < E; e += blockDim.x) off[e] = cnt[e] > 0 ? 1 : 0;
    __syncthreads();
    const int n_active = block_exclusive_scan(off, E);
    for (int e = tid; e < E; e += blockDim.x)
        if (cnt[e] > 0) active[off[e]] = e;
    if (tid == 0) active[E] = n_active;
}

// Logits by GEMV (one warp per expert, all T tokens), then the last CTA to
// finish runs top-k for every token and, if requested, the permutation.
// Each warp issues all loads of its weight row before it needs them; the T
// token rows are staged once per CTA in shared memory.  With xq requested,
// the CTAs also write the rows as E2M1 terms for the expert kernels.
constexpr int kRouteChunks = 16;  // 16-byte weight loads per lane in flight

__global__ void __launch_bounds__(256)
route_small_kernel(RouteArgs a) {
    extern __shared__ __align__(16) uint4 xs[];  // [T * d_r / 8]
    __shared__ int32_t sel[256];
    __shared__ uint32_t ticket_s;
    // the next kernel of the forward may start launching now: it waits for
    // this grid's completion (griddepcontrol.wait) before reading its outputs
    pdl_trigger();
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int e = blockIdx.x * 8 + wid;
    const uint16_t* wrow = a.w + static_cast<size_t>(e < a.E ? e : 0) * a.d_r;
    uint4 wv[kRouteChunks];
#pragma unroll
    for (int i = 0; i < kRouteChunks; ++i) {
        const int c = i * 256 + lane * 8;
        wv[i] = (e < a.E && c < a.d_r) ? ldg_nc_v4(wrow + c) : make_uint4(0, 0, 0, 0);
    }
    const int nvec = a.T * a.d_r / 8;
    for (int v = threadIdx.x; v < nvec; v += blockDim.x)
        xs[v] = reinterpret_cast<const uint4*>(a.x)[v];
    __syncthreads();

    // router input -> E2M1 terms for the block-scaled expert kernels: one warp
    // per 32-element block, blocks spread over all warps of the grid (the
    // rows are staged in every CTA)
    if (a.xq) {
        const int nb = a.d_r / 32;
        for (int i = blockIdx.x * 8 + wid; i < a.T * nb; i += gridDim.x * 8) {
            const int t = i / nb, b = i - t * nb;
            const uint16_t* row = reinterpret_cast<const uint16_t*>(xs) + static_cast<size_t>(t) * a.d_r;
            uint32_t q[kTerms], sb[kTerms];
            quantize_terms(bf16_to_f32(row[32 * b + lane]), q, sb);
            store_terms(q, sb, t, b & 7, a.xq + static_cast<size_t>(b >> 3) * a.xq_n * 128,
                        a.xsf + static_cast<size_t>(b >> 3) * 1024);
        }
    }

    if (e < a.E) {
        float acc[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) acc[t] = 0.0f;
        for (int base = 0; base < a.d_r; base += 256 * kRouteChunks) {
            if (base > 0) {
#pragma unroll
                for (int i = 0; i < kRouteChunks; ++i) {
                    const int c = base + i * 256 + lane * 8;
                    wv[i] = c < a.d_r ? ldg_nc_v4(wrow + c) : make_uint4(0, 0, 0, 0);
                }
            }
#pragma unroll
            for (int i = 0; i < kRouteChunks; ++i) {
                const int c = base + i * 256 + lane * 8;
                if (c >= a.d_r) break;
                const uint32_t wq[4] = {wv[i].x, wv[i].y, wv[i].z, wv[i].w};
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    if (t >= a.T) break;
                    const uint4 xv = xs[(t * a.d_r + c) / 8];
                    const uint32_t xq[4] = {xv.x, xv.y, xv.z, xv.w};
                    float sacc = acc[t];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        sacc = fmaf(__uint_as_float(wq[q] << 16), __uint_as_float(xq[q] << 16), sacc);
                        sacc = fmaf(__uint_as_float(wq[q] & 0xFFFF0000u),
                                    __uint_as_float(xq[q] & 0xFFFF0000u), sacc);
                    }
                    acc[t] = sacc;
                }
            }
        }
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            if (t >= a.T) break;
            const float v = warp_sum(acc[t]);
            if (lane == 0) a.logits[static_cast<size_t>(t) * a.E + e] = v;
        }
    }
    // last CTA to finish does the selection
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) ticket_s = atomicAdd(&a.hdr->counters[CTR_ROUTE], 1u);
    __syncthreads();
    if (ticket_s != gridDim.x - 1) return;
    if (threadIdx.x == 0) a.hdr->counters[CTR_ROUTE] = 0;
    __threadfence();
    {
        __shared__ uint64_t cand[8][32];
        if (a.T == 1) topk_tokens_cta<8>(a, sel, cand);
        else if (a.T == 2) topk_tokens_cta<4>(a, sel, cand);
        else if (a.T <= 4) topk_tokens_cta<2>(a, sel, cand);
        else topk_tokens_cta<1>(a, sel, cand);
    }
    __syncthreads();
    if (a.counts)
        permute_small(sel, a.T, a.k, a.E, a.counts, a.offsets, a.perm, a.inv, a.active);
}

__global__ void __launch_bounds__(256)
topk_kernel(RouteArgs a) {
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= a.T) return;
    topk_token(a.logits + static_cast<size_t>(t) * a.E, a.bias, a.E, a.k,
               a.idx + static_cast<size_t>(t) * a.k, a.wts + static_cast<size_t>(t) * a.k,
               nullptr, a.hdr);
}

// Plain tiled SIMT logits for moderate T: 64 tokens x 64 experts per CTA.
__global__ void __launch_bounds__(256)
logits_simt_kernel(RouteArgs a) {
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
perm_count_kernel(const int32_t* __restrict__ idx, int T, int k, int E, int32_t* chunk_cnt,
                  WsHeader* hdr) {
    extern __shared__ int hist[];
    const int c = blockIdx.x;
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    const int t0 = c * kChunk, t1 = min(T, t0 + kChunk);
    for (int p = t0 * k + threadIdx.x; p < t1 * k; p += blockDim.x) {
        const int e = idx[p];
        if (e >= 0 && e < E)
            atomicAdd(&hist[e], 1);
        else
            set_error(hdr, K3MOE_ERR_INVALID_ARG, 2);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        chunk_cnt[static_cast<size_t>(c) * E + e] = hist[e];
}

// one CTA: per-expert running sums over chunks, exclusive scan over experts,
// active list
__global__ void __launch_bounds__(256)
perm_scan_kernel(int32_t* chunk_cnt, int nchunks, int E, int P, int32_t* counts,
                 int32_t* offsets, int32_t* active) {
    extern __shared__ int sm[];  // [2 * E]
    int* tot = sm;
    int* flag = sm + E;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = 0;
        for (int c = 0; c < nchunks; ++c) {
            int* p = chunk_cnt + static_cast<size_t>(c) * E + e;
            const int v = *p;
            *p = run;  // exclusive within the expert
            run += v;
        }
        tot[e] = run;
        counts[e] = run;
        flag[e] = run > 0 ? 1 : 0;
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
                    int32_t* perm, int32_t* inv) {
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

cudaError_t launch_route_small(const RouteArgs& a, cudaStream_t s) {
    const int grid = (a.E + 7) / 8;
    const size_t smem = static_cast<size_t>(a.T) * a.d_r * 2;
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(route_small_kernel,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    route_small_kernel<<<grid, 256, smem, s>>>(a);
    trace_mark("route_small", s);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Router with library-owned scratch (k3moe_route_noalloc).
//
// The small-T router needs a completion counter and, when the caller does
// not want the logits, a [T, E] fp32 buffer for them.  This variant keeps
// both in one file-scope device array instead of a caller workspace: it is
// part of the module image, so every GPU that loads the library holds these
// bytes until the process exits, and every call shares them.
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
    a.counts = nullptr;
    return launch_route_small(a, s);
}

cudaError_t launch_topk(const RouteArgs& a, cudaStream_t s) {
    topk_kernel<<<(a.T + 7) / 8, 256, 0, s>>>(a);
    trace_mark("topk", s);
    return cudaGetLastError();
}

cudaError_t launch_logits_simt(const RouteArgs& a, cudaStream_t s) {
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
                           void* scratch, WsHeader* hdr, cudaStream_t s) {
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
    perm_count_kernel<<<nchunks, 256, smem, s>>>(idx, T, k, E, chunk, hdr);
    trace_mark("perm_count", s);
    perm_scan_kernel<<<1, 256, 2 * smem, s>>>(chunk, nchunks, E, T * k, counts, offsets, active);
    trace_mark("perm_scan", s);
    perm_scatter_kernel<<<nchunks, 32, smem, s>>>(idx, T, k, E, chunk, offsets, perm, inv);
    trace_mark("perm_scatter", s);
    return cudaGetLastError();
}

}  // namespace k3
