// Device cache of host-resident experts.
//
// The expert weights stay in host memory (page-locked and mapped into the
// device address space; on GB300 the GPU reads it over NVLink-C2C) and a
// fixed number of expert slots in HBM holds the recently used experts.  Every
// call, after the router has listed the experts its tokens use (the union over
// the call's tokens, so a batch of draft tokens fetches each expert once), one
// CTA assigns slots: used experts already resident are hits and have their
// slot's stamp refreshed; the missing ones take the least recently used slots
// that this call does not use.  Then every SM copies the missing experts'
// codes and scale atoms from host memory into their slots, and the streaming
// expert kernels read the weights through the expert -> slot map.
//
// The policy follows the deployment that the K3-Stuff page ("llama-cpp-
// patches", change 2) describes, where the page cache serves as the hot-expert
// cache with lazy fault-in and least-recently-used eviction; the Lucebox PR
// #573 page ("Runtime validation") runs the same model with an 8 GiB device
// expert cache and route-batched verification.  Here the host tier is pinned
// memory instead of a file, and the slots are stamped per call: every expert
// a call uses counts as used at the same time.  Victims are the slots with the
// oldest stamps (never-used slots first); among equal stamps the lower slot
// index goes first, and the i-th missing expert (ascending expert index) takes
// the i-th victim (ascending slot index).  The assignment is integer work and
// deterministic.
#include "common.cuh"

namespace k3 {

namespace {

constexpr int kAssignThreads = 1024;
constexpr int kFillThreads = 256;
constexpr int kFillVec = 4;                                   // 16-byte loads in flight per thread
constexpr uint32_t kPiece = kFillThreads * kFillVec * 16;     // bytes per CTA pass (16 KB)

// exclusive prefix sum of v over the block's threads; *total = the block's sum
__device__ int block_scan_excl(int v, int* total) {
    __shared__ int wsum[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int x = v;
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nw ? wsum[lane] : 0;
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        wsum[lane] = w;
    }
    __syncthreads();
    const int before = (warp ? wsum[warp - 1] : 0) + x - v;
    *total = wsum[nw - 1];
    __syncthreads();
    return before;
}

__global__ void __launch_bounds__(256) cache_init_kernel(CacheView c, int E, int S) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < E) c.slot_of[i] = -1;
    if (i < S) {
        c.expert_of[i] = -1;
        c.stamp[i] = 0;
        c.miss_e[i] = -1;
        c.miss_slot[i] = -1;
    }
    if (i == 0) {
        CacheHeader h{};
        h.magic = kCacheMagic;
        h.E = E;
        h.slots = S;
        *c.h = h;
    }
}

// one CTA; E <= 1024 and S <= E
__global__ void __launch_bounds__(kAssignThreads)
cache_assign_kernel(CacheView c, int E, int S, const int32_t* __restrict__ active,
                    unsigned long long expert_bytes, WsHeader* hdr) {
    __shared__ int victim[kAssignThreads];
    __shared__ int s_bad;
    pdl_wait();     // the active list is final
    pdl_trigger();  // the copy kernel waits for this grid to complete
    const int t = threadIdx.x;
    CacheHeader* h = c.h;
    if (t == 0) {
        int bad = (h->magic != kCacheMagic || h->E != E || h->slots != S) ? 1 : 0;
        const int U = bad ? 0 : active[E];
        if (!bad && (U < 0 || U > E || U > S)) bad = 2;
        s_bad = bad;
        if (bad) {
            set_error(hdr, K3MOE_ERR_INVALID_ARG, 80 + bad);
            h->last_miss = 0;
        }
    }
    __syncthreads();
    if (s_bad) return;
    const uint32_t clock = h->clock + 1;
    const int U = active[E];

    // hits: refresh the stamp of every used, resident expert
    int e = -1, hit = 0;
    if (t < U) {
        e = active[t];
        if (e < 0 || e >= E) {
            set_error(hdr, K3MOE_ERR_INVALID_ARG, 83);
            e = -1;
        } else {
            const int s = c.slot_of[e];
            if (s >= 0 && s < S) {
                hit = 1;
                c.stamp[s] = clock;
            }
        }
    }
    const int miss = (e >= 0 && !hit) ? 1 : 0;
    int m_all;
    const int mr = block_scan_excl(miss, &m_all);  // its barriers publish the stamps
    if (miss) c.miss_e[mr] = e;

    // victims: the m least recently used slots that this call does not use
    uint32_t key = 0;
    int valid = 0;
    if (t < S) {
        key = c.stamp[t];
        valid = key != clock;
    }
    int m = m_all;
    uint32_t lo = 0, hi = clock - 1;  // the keys of valid slots are below clock
    if (m > 0) {
        const int avail = __syncthreads_count(valid);
        if (avail < m) {
            if (t == 0) set_error(hdr, K3MOE_ERR_INVALID_ARG, 84);
            m = avail;
        }
        while (lo < hi) {  // smallest tau with #{valid, key <= tau} >= m
            const uint32_t mid = lo + (hi - lo) / 2;
            if (__syncthreads_count(valid && key <= mid) >= m)
                hi = mid;
            else
                lo = mid + 1;
        }
    }
    const uint32_t tau = lo;
    const int less = __syncthreads_count(valid && key < tau);
    int eq_total;
    const int eq_rank = block_scan_excl((valid && key == tau) ? 1 : 0, &eq_total);
    const int vict = (m > 0 && valid && (key < tau || (key == tau && eq_rank < m - less))) ? 1 : 0;
    int v_total;
    const int v_rank = block_scan_excl(vict, &v_total);
    if (vict) victim[v_rank] = t;
    __syncthreads();

    if (t < m) {
        const int v = victim[t], ne = c.miss_e[t];
        const int old = c.expert_of[v];
        if (old >= 0 && old < E) c.slot_of[old] = -1;  // not used by this call: its stamp is older
        c.expert_of[v] = ne;
        c.slot_of[ne] = v;
        c.stamp[v] = clock;
        c.miss_slot[t] = v;
    }
    if (t == 0) {
        h->clock = clock;
        h->last_miss = m;
        h->last_hit = U - m_all;
        h->calls += 1;
        h->hits += static_cast<unsigned long long>(U - m_all);
        h->misses += static_cast<unsigned long long>(m);
        h->bytes += static_cast<unsigned long long>(m) * expert_bytes;
    }
}

__device__ __forceinline__ const uint8_t* pick(const uint8_t* const (&p)[3], uint32_t i) {
    return i == 0 ? p[0] : (i == 1 ? p[1] : p[2]);
}
__device__ __forceinline__ uint8_t* pick(uint8_t* const (&p)[3], uint32_t i) {
    return i == 0 ? p[0] : (i == 1 ? p[1] : p[2]);
}

// every CTA copies 16 KB pieces of the missing experts (codes, then scale
// atoms, of w1, w3 and w2) from host memory into their slots
__global__ void __launch_bounds__(kFillThreads)
cache_fill_kernel(CacheView c, CacheFillArgs a) {
    pdl_wait();     // the slot assignment is final
    pdl_trigger();  // the expert kernels wait for this grid to complete
    const uint32_t m = static_cast<uint32_t>(max(c.h->last_miss, 0));
    const uint32_t cq = static_cast<uint32_t>((a.q_bytes + kPiece - 1) / kPiece);
    const uint32_t cs = static_cast<uint32_t>((a.sf_bytes + kPiece - 1) / kPiece);
    const uint32_t per = 3 * (cq + cs);
    const uint32_t total = per * m;
    for (uint32_t w = blockIdx.x; w < total; w += gridDim.x) {
        const uint32_t i = w / per;
        uint32_t r = w - i * per;
        const size_t e = static_cast<size_t>(c.miss_e[i]), v = static_cast<size_t>(c.miss_slot[i]);
        const uint8_t* src;
        uint8_t* dst;
        size_t n;
        if (r < 3 * cq) {
            const uint32_t mat = r / cq;
            const size_t off = static_cast<size_t>(r - mat * cq) * kPiece;
            n = min(static_cast<size_t>(kPiece), a.q_bytes - off);
            src = pick(a.src_q, mat) + e * a.q_bytes + off;
            dst = pick(a.dst_q, mat) + v * a.q_bytes + off;
        } else {
            r -= 3 * cq;
            const uint32_t mat = r / cs;
            const size_t off = static_cast<size_t>(r - mat * cs) * kPiece;
            n = min(static_cast<size_t>(kPiece), a.sf_bytes - off);
            src = pick(a.src_sf, mat) + e * a.sf_bytes + off;
            dst = pick(a.dst_sf, mat) + v * a.sf_bytes + off;
        }
        const uint4* s4 = reinterpret_cast<const uint4*>(src);
        uint4* d4 = reinterpret_cast<uint4*>(dst);
        const int nv = static_cast<int>(n / 16);
        uint4 x[kFillVec];
#pragma unroll
        for (int j = 0; j < kFillVec; ++j) {
            const int k = threadIdx.x + j * kFillThreads;
            if (k < nv) x[j] = s4[k];
        }
#pragma unroll
        for (int j = 0; j < kFillVec; ++j) {
            const int k = threadIdx.x + j * kFillThreads;
            if (k < nv) d4[k] = x[j];
        }
    }
}

}  // namespace

size_t cache_state_bytes(int E, int slots) {
    return sizeof(CacheHeader) + align_up(static_cast<size_t>(E) * 4) + 4 * align_up(static_cast<size_t>(slots) * 4);
}

CacheView cache_view(void* state, int E, int slots) {
    char* b = static_cast<char*>(state);
    CacheView c;
    size_t o = sizeof(CacheHeader);
    c.h = reinterpret_cast<CacheHeader*>(b);
    c.slot_of = reinterpret_cast<int32_t*>(b + o);
    o += align_up(static_cast<size_t>(E) * 4);
    c.expert_of = reinterpret_cast<int32_t*>(b + o);
    o += align_up(static_cast<size_t>(slots) * 4);
    c.stamp = reinterpret_cast<uint32_t*>(b + o);
    o += align_up(static_cast<size_t>(slots) * 4);
    c.miss_e = reinterpret_cast<int32_t*>(b + o);
    o += align_up(static_cast<size_t>(slots) * 4);
    c.miss_slot = reinterpret_cast<int32_t*>(b + o);
    return c;
}

cudaError_t launch_cache_init(void* state, int E, int slots, cudaStream_t s) {
    const int n = E > slots ? E : slots;
    cache_init_kernel<<<(n + 255) / 256, 256, 0, s>>>(cache_view(state, E, slots), E, slots);
    return cudaGetLastError();
}

cudaError_t launch_cache_update(void* state, int E, int slots, const int32_t* active,
                                const CacheFillArgs& f, WsHeader* hdr, int num_sms, cudaStream_t s) {
    if (E > kAssignThreads || slots > E) return cudaErrorNotSupported;
    const CacheView c = cache_view(state, E, slots);
    const unsigned long long expert_bytes = 3ull * (f.q_bytes + f.sf_bytes);
    cudaError_t e = launch_pdl(cache_assign_kernel, dim3(1), dim3(kAssignThreads), 0, s, c, E, slots, active,
                               expert_bytes, hdr);
    trace_mark("cache_assign", s);
    if (e != cudaSuccess) return e;
    e = launch_pdl(cache_fill_kernel, dim3(8 * num_sms), dim3(kFillThreads), 0, s, c, f);
    trace_mark("cache_fill", s);
    return e;
}

}  // namespace k3
