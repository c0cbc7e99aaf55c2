// Decode path (T <= 8): the expert FFN as streaming GEMVs over the bytes of
// the selected experts only.  Token-generation time in the pages goes into
// reading routed-expert bytes (llama.cpp PR #26185 "model: add Kimi-K3 text
// model"; Lucebox PR #573, SSD-routed expert payloads), so these kernels are
// built to keep HBM busy: every weight byte of a selected expert is read once,
// with 16-byte loads that cover whole 64-byte runs of a row, several chunks in
// flight per warp, and an even split of the bytes over all warps.
//
// Arithmetic (fp32 accumulation).  A warp owns 16 weight rows and up to 8
// token rows and uses the register-operand MMA m16n8k16 (f16 x f16 -> fp32):
//   * A fragment: the lane (g, t) loads the 16 bytes of block 4c + t of rows
//     g and g + 8 (one 32-element E2M1 block each), converts them exactly to
//     f16 (cvt e2m1x2) and multiplies by 2^(e_b - e_ref), where e_b is the
//     block's E8M0 exponent and e_ref the largest exponent of the row's four
//     blocks in this chunk (an exact power of two in f16);
//   * the 16-wide K slice of MMA j takes elements 4j..4j+3 of each lane's
//     block; B uses the same mapping, so lane (g, t) reads elements 4j..4j+3
//     of block 4c + t of token g: a permutation of the reduction order only;
//   * activations are f16 with one power-of-two exponent per token row
//     (x * 2^-e_x, |x * 2^-e_x| < 2), applied back in fp32;
//   * the chunk's fp32 sums are scaled by 2^(e_ref - 127) and accumulated in
//     fp32.
// Work split: the units (selected expert, 16-row tile, 128-wide K chunk) are
// cut into equal contiguous ranges, one per warp, each at least one tile
// long, so a tile is shared by at most two warps.  Each writes its partial sum
// to its own slot (0 for the warp that starts the tile, 1 for the other; a
// warp that owns the whole tile writes zero to slot 1); the consumer adds
// slot 0 and slot 1 in that order, so results are deterministic.
//
// Kernels: prep (f16 token rows), up (w1/w3 partial sums), finish_up (h =
// silu(g) * u in fp32, then f16 with a per-row exponent), down (w2 partial
// sums), combine (slot order).
#include "common.cuh"

namespace k3 {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxTok = 8;   // tokens per expert (N of the MMA)

__device__ __forceinline__ float silu_f32(float g) { return g / (1.0f + expf(-g)); }

// d += A * B on the register-operand MMA m16n8k16 (f16 inputs, fp32 accumulator)
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void convert_scaled(const uint4& raw, uint32_t sc2, uint32_t (&w)[16]) {
    e2m1x8_to_f16x8(raw.x, w[0], w[1], w[2], w[3]);
    e2m1x8_to_f16x8(raw.y, w[4], w[5], w[6], w[7]);
    e2m1x8_to_f16x8(raw.z, w[8], w[9], w[10], w[11]);
    e2m1x8_to_f16x8(raw.w, w[12], w[13], w[14], w[15]);
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = hmul2(w[i], sc2);
}

struct Phase {
    const uint8_t* q[2];     // packed E2M1 of the (one or two) matrices [E * rows, K / 2]
    const uint8_t* s[2];     // E8M0 [E * rows, K / 32]
    int nmat;
    int rows;                // rows of one expert matrix
    int K;
    const uint16_t* b;       // f16 token rows: [T, K] (by token) or [P, K] (by pair row)
    const int32_t* bexp;     // per row of b
    int b_by_token;          // 1: b row = token of the pair; 0: b row = pair row
    float* part;             // [nmat][2 slots][P][rows]
    int P;
};

constexpr int kStages = 4;      // chunks in flight per warp (cp.async ring)
constexpr int kTileTab = 16;    // tile descriptors cached per warp

// Per-warp shared memory: the ring (weight cells, scale words) and the table
// of tile descriptors of the warp's range.
template <int NMAT>
struct WarpSmem {
    uint4 w[kStages][NMAT][2][32];      // lane's 16 bytes of rows g / g+8
    uint32_t sc[kStages][NMAT][2][32];  // lane's scale word (blocks 4c..4c+3) of rows g / g+8
    int tab_e[kTileTab];                // expert
    int tab_o0[kTileTab];               // first pair row of the expert
    int tab_n[kTileTab];                // tokens of the expert (<= 8)
    int tab_rt[kTileTab];               // 16-row tile of the matrix
    int tab_brow[kTileTab][kMaxTok];    // b row of each token slot
};

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}

__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// max of the four bytes of w
__device__ __forceinline__ int max4_bytes(uint32_t w) {
    uint32_t m = __vmaxu4(w, w >> 16);
    m = __vmaxu4(m, m >> 8);
    return static_cast<int>(m & 0xFF);
}

// Stream-K phase: partial sums of (selected expert, 16-row tile) over each warp's
// contiguous share of the (tile, 128-wide K chunk) units.  The weight bytes of
// a unit are copied with cp.async into a per-warp ring kStages - 1 units ahead
// of the math, across tile boundaries.
template <int NMAT>
__global__ void __launch_bounds__(kThreads)
decode_phase_kernel(DecodeArgs a, Phase ph) {
    extern __shared__ __align__(16) unsigned char dsmem[];
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int g = lane >> 2, t = lane & 3;
    WarpSmem<NMAT>& sm = reinterpret_cast<WarpSmem<NMAT>*>(dsmem)[wid];
    const int64_t warp = static_cast<int64_t>(blockIdx.x) * kWarps + wid;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;
    const int U = a.active[a.E];
    const int R = ph.rows / 16;
    const int C = (ph.K + 127) / 128;
    const int nb = ph.K / 32;
    const bool scale_words = (nb & 3) == 0;
    const size_t kq = static_cast<size_t>(ph.K / 2);
    const int n_tiles = U * R;
    const int64_t W = static_cast<int64_t>(n_tiles) * C;
    const int64_t G = nwarps < n_tiles ? nwarps : n_tiles;  // each range >= one tile
    if (warp >= G) return;
    // this warp's units [start, end); 32-bit counters from here on
    const int start = static_cast<int>(W * warp / G), end = static_cast<int>(W * (warp + 1) / G);
    const int tile_first = start / C;

    // table of tile descriptors for tiles tile_first + [tab0, tab0 + kTileTab)
    int tab0 = -1;
    auto fill_table = [&](int base) {
        __syncwarp();
        if (lane < kTileTab) {
            const int tile = tile_first + base + lane;
            if (tile < n_tiles) {
                const int au = tile / R;
                const int e = a.active[au];
                const int o0 = a.offsets[e];
                const int n = min(a.offsets[e + 1] - o0, kMaxTok);
                sm.tab_e[lane] = e;
                sm.tab_o0[lane] = o0;
                sm.tab_n[lane] = n;
                sm.tab_rt[lane] = tile - au * R;
                for (int j = 0; j < kMaxTok; ++j)
                    sm.tab_brow[lane][j] = j < n ? (ph.b_by_token ? a.perm[o0 + j] / a.k : o0 + j) : 0;
            }
        }
        __syncwarp();
        tab0 = base;
    };
    // table slot of a tile, refilling as needed.  The issue side runs at most
    // kStages - 1 units (so at most kStages tiles) ahead of the math side, and
    // the math side copies what it needs into registers when it enters a tile,
    // so a refill keeps kStages tiles of margin behind the requested one.
    auto slot_of = [&](int tile) -> int {
        const int rel = tile - tile_first;
        if (tab0 < 0 || rel < tab0 || rel >= tab0 + kTileTab)
            fill_table(rel > kStages ? rel - kStages : 0);
        return rel - tab0;
    };

    // issue the copies of unit (tile, c) into ring stage st
    auto issue = [&](int tile, int c, int st) {
        const int ts = slot_of(tile);
        const size_t row0 = static_cast<size_t>(sm.tab_e[ts]) * ph.rows + sm.tab_rt[ts] * 16 + g;
        const int blk = 4 * c + t;
        const bool ok = blk < nb;
#pragma unroll
        for (int m = 0; m < NMAT; ++m) {
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const size_t row = row0 + 8 * r;
                cp_async16(&sm.w[st][m][r][lane], ph.q[m] + row * kq + (ok ? 16 * blk : 0), ok);
                if (scale_words) cp_async4(&sm.sc[st][m][r][lane], ph.s[m] + row * nb + 4 * c);
            }
        }
    };

    // issue side: next unit to copy, as (tile, chunk, ring stage)
    int it_tile = start / C, it_c = start - (start / C) * C, it_st = 0;
    int issued = start;
    auto issue_next = [&]() {
        if (issued < end) issue(it_tile, it_c, it_st);
        cp_async_commit();
        ++issued;
        if (++it_c == C) { it_c = 0; ++it_tile; }
        it_st = (it_st + 1) & (kStages - 1);
    };
    // prologue: kStages - 1 units in flight
#pragma unroll
    for (int i = 0; i < kStages - 1; ++i) issue_next();

    float tot[NMAT][4];
    int cur_tile = -1;
    int n = 0, o0 = 0, rt = 0, c0 = 0;
    int bq[2] = {0, 0};  // b rows of tokens 2t, 2t+1 (for their exponents)
    size_t row0 = 0;
    const uint16_t* brow = ph.b;
    bool has_tok = false;
    uint4 xr[4];

    auto flush = [&](int c_end) {
        // write the partial sums of tokens 2t, 2t+1 (rows g, g+8)
        const int slot = c0 == 0 ? 0 : 1;
        const bool whole = c0 == 0 && c_end == C;
        const int r0 = rt * 16 + g;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int tok = 2 * t + q;
            if (tok >= n) continue;
            const int pr = o0 + tok;
            const float sx = exp2i(ph.bexp[bq[q]]);
#pragma unroll
            for (int m = 0; m < NMAT; ++m) {
                float* base = ph.part + (static_cast<size_t>(m) * 2) * ph.P * ph.rows;
                float* p0 = base + static_cast<size_t>(slot) * ph.P * ph.rows + static_cast<size_t>(pr) * ph.rows;
                p0[r0] = tot[m][q] * sx;
                p0[r0 + 8] = tot[m][2 + q] * sx;
                if (whole) {
                    float* p1 = base + static_cast<size_t>(ph.P) * ph.rows + static_cast<size_t>(pr) * ph.rows;
                    p1[r0] = 0.0f;
                    p1[r0 + 8] = 0.0f;
                }
            }
        }
    };

    int tile = start / C, c = start - (start / C) * C, st = 0;
    for (int u = start; u < end; ++u) {
        issue_next();  // keeps kStages - 1 units in flight
        if (tile != cur_tile) {
            if (cur_tile >= 0) flush(C);
            cur_tile = tile;
            const int ts = slot_of(tile);
            n = sm.tab_n[ts];
            o0 = sm.tab_o0[ts];
            rt = sm.tab_rt[ts];
            c0 = c;
            row0 = static_cast<size_t>(sm.tab_e[ts]) * ph.rows + rt * 16 + g;
            has_tok = g < n;
            brow = ph.b + static_cast<size_t>(sm.tab_brow[ts][has_tok ? g : 0]) * ph.K;
            bq[0] = sm.tab_brow[ts][min(2 * t, kMaxTok - 1)];
            bq[1] = sm.tab_brow[ts][min(2 * t + 1, kMaxTok - 1)];
#pragma unroll
            for (int m = 0; m < NMAT; ++m) tot[m][0] = tot[m][1] = tot[m][2] = tot[m][3] = 0.0f;
        }
        // token block of x (f16), zero beyond the tokens / blocks
        const int blk = 4 * c + t;
        if (has_tok && blk < nb) {
            const uint4* xb = reinterpret_cast<const uint4*>(brow + 32 * blk);
#pragma unroll
            for (int i = 0; i < 4; ++i) xr[i] = xb[i];
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) xr[i] = make_uint4(0, 0, 0, 0);
        }
        cp_async_wait<kStages - 1>();  // unit u's copies (this lane's) have landed

        const uint32_t xw[16] = {xr[0].x, xr[0].y, xr[0].z, xr[0].w, xr[1].x, xr[1].y,
                                 xr[1].z, xr[1].w, xr[2].x, xr[2].y, xr[2].z, xr[2].w,
                                 xr[3].x, xr[3].y, xr[3].z, xr[3].w};
#pragma unroll
        for (int m = 0; m < NMAT; ++m) {
            uint32_t sw0, sw8;
            if (scale_words) {
                sw0 = sm.sc[st][m][0][lane];
                sw8 = sm.sc[st][m][1][lane];
            } else {
                sw0 = sw8 = 0;
                for (int b = 0; b < 4; ++b)
                    if (4 * c + b < nb) {
                        sw0 |= static_cast<uint32_t>(__ldg(ph.s[m] + row0 * nb + 4 * c + b)) << (8 * b);
                        sw8 |= static_cast<uint32_t>(__ldg(ph.s[m] + (row0 + 8) * nb + 4 * c + b)) << (8 * b);
                    }
            }
            const int er0 = max4_bytes(sw0), er8 = max4_bytes(sw8);
            const uint32_t h0 = f16_pow2(static_cast<int>((sw0 >> (8 * t)) & 0xFF) - er0);
            const uint32_t h8 = f16_pow2(static_cast<int>((sw8 >> (8 * t)) & 0xFF) - er8);
            uint32_t w0[16], w8[16];
            convert_scaled(sm.w[st][m][0][lane], h0 | (h0 << 16), w0);
            convert_scaled(sm.w[st][m][1][lane], h8 | (h8 << 16), w8);
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < 8; ++j)
                mma16816(acc, w0[2 * j], w8[2 * j], w0[2 * j + 1], w8[2 * j + 1], xw[2 * j], xw[2 * j + 1]);
            const float s0 = exp2i(er0 - 127), s8 = exp2i(er8 - 127);
            tot[m][0] = fmaf(acc[0], s0, tot[m][0]);
            tot[m][1] = fmaf(acc[1], s0, tot[m][1]);
            tot[m][2] = fmaf(acc[2], s8, tot[m][2]);
            tot[m][3] = fmaf(acc[3], s8, tot[m][3]);
        }
        const bool last_of_tile = (c == C - 1) || (u + 1 == end);
        if (last_of_tile) {
            flush(c + 1);
            cur_tile = -1;
        }
        if (++c == C) { c = 0; ++tile; }
        st = (st + 1) & (kStages - 1);
    }
    cp_async_wait<0>();
}

template <int NMAT>
constexpr size_t phase_smem() { return sizeof(WarpSmem<NMAT>) * kWarps; }

// token rows -> f16 with one exponent per row (one warp per row)
__global__ void __launch_bounds__(256)
prep_rows_kernel(const uint16_t* __restrict__ x, int T, int K, uint16_t* __restrict__ x16,
                 int32_t* __restrict__ xexp) {
    pdl_wait();
    pdl_trigger();
    const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (r >= T) return;
    const int ex = row_to_f16(x + static_cast<size_t>(r) * K, K, x16 + static_cast<size_t>(r) * K);
    if ((threadIdx.x & 31) == 0) xexp[r] = ex;
}

// h = silu(g) * u from the two partial slots (slot 0 + slot 1), then f16 with a
// per-row exponent.  One CTA per pair row; every thread loads its elements
// with independent 16-byte loads, so the row costs two memory round trips.
constexpr int kFinishThreads = 256;
constexpr int kFinishPerThread = 16;  // f <= 4096

__global__ void __launch_bounds__(kFinishThreads)
finish_up_kernel(const float* __restrict__ part, int P, int f, uint16_t* __restrict__ h16,
                 int32_t* __restrict__ hexp) {
    __shared__ float wmax[kFinishThreads / 32];
    pdl_wait();
    pdl_trigger();
    const int p = blockIdx.x;
    const size_t plane = static_cast<size_t>(P) * f;
    const float* g0 = part + static_cast<size_t>(p) * f;
    float h[kFinishPerThread];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < kFinishPerThread / 4; ++i) {
        const int c = (i * kFinishThreads + threadIdx.x) * 4;
        if (c < f) {
            const float4 a0 = *reinterpret_cast<const float4*>(g0 + c);
            const float4 a1 = *reinterpret_cast<const float4*>(g0 + plane + c);
            const float4 b0 = *reinterpret_cast<const float4*>(g0 + 2 * plane + c);
            const float4 b1 = *reinterpret_cast<const float4*>(g0 + 3 * plane + c);
            h[4 * i + 0] = silu_f32(a0.x + a1.x) * (b0.x + b1.x);
            h[4 * i + 1] = silu_f32(a0.y + a1.y) * (b0.y + b1.y);
            h[4 * i + 2] = silu_f32(a0.z + a1.z) * (b0.z + b1.z);
            h[4 * i + 3] = silu_f32(a0.w + a1.w) * (b0.w + b1.w);
#pragma unroll
            for (int j = 0; j < 4; ++j) amax = fmaxf(amax, fabsf(h[4 * i + j]));
        }
    }
    amax = warp_max(amax);
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = amax;
    __syncthreads();
    float m = 0.0f;
#pragma unroll
    for (int w = 0; w < kFinishThreads / 32; ++w) m = fmaxf(m, wmax[w]);
    const int ex = ilog2f(m);
    const float sc = exp2i(-ex);
    uint16_t* dst = h16 + static_cast<size_t>(p) * f;
#pragma unroll
    for (int i = 0; i < kFinishPerThread / 4; ++i) {
        const int c = (i * kFinishThreads + threadIdx.x) * 4;
        if (c < f) {
            uint2 o;
            o.x = f32x2_to_f16x2(h[4 * i] * sc, h[4 * i + 1] * sc);
            o.y = f32x2_to_f16x2(h[4 * i + 2] * sc, h[4 * i + 3] * sc);
            *reinterpret_cast<uint2*>(dst + c) = o;
        }
    }
    if (threadIdx.x == 0) hexp[p] = ex;
}

template <int NMAT>
cudaError_t launch_phase(const DecodeArgs& a, const Phase& ph, cudaStream_t s, const char* name) {
    // four CTAs of four warps per SM; the kernel trims the warp count so that
    // every warp owns at least one whole tile of K chunks
    const int grid = 4 * a.num_sms;
    constexpr size_t smem = phase_smem<NMAT>();
    static bool attr_set = false;  // per process; one GPU per process here
    if (!attr_set) {
        cudaFuncSetAttribute(decode_phase_kernel<NMAT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
        attr_set = true;
    }
    const cudaError_t e = launch_pdl(decode_phase_kernel<NMAT>, dim3(grid), dim3(kThreads), smem, s, a, ph);
    trace_mark(name, s);
    return e;
}

}  // namespace

size_t decode_scratch_bytes(int T, int k, int d, int f) {
    const size_t P = static_cast<size_t>(T) * k;
    size_t b = 0;
    b += align_up(static_cast<size_t>(T) * d * 2);      // x16
    b += align_up(static_cast<size_t>(T) * 4);          // xexp
    b += align_up(4 * P * f * 4);                        // up partials [2 mats][2 slots][P][f]
    b += align_up(P * f * 2);                            // h16
    b += align_up(P * 4);                                // hexp
    return b;
}

void decode_x16_slots(void* scratch, int T, int d, uint16_t** x16, int32_t** xexp) {
    char* base = static_cast<char*>(scratch);
    *x16 = reinterpret_cast<uint16_t*>(base);
    *xexp = reinterpret_cast<int32_t*>(base + align_up(static_cast<size_t>(T) * d * 2));
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
    const int P = a.T * a.k;
    char* base = reinterpret_cast<char*>(a.scratch);
    uint16_t* x16 = reinterpret_cast<uint16_t*>(base);
    base += align_up(static_cast<size_t>(a.T) * a.d * 2);
    int32_t* xexp = reinterpret_cast<int32_t*>(base);
    base += align_up(static_cast<size_t>(a.T) * 4);
    float* upart = reinterpret_cast<float*>(base);
    base += align_up(4ull * P * a.f * 4);
    uint16_t* h16 = reinterpret_cast<uint16_t*>(base);
    base += align_up(static_cast<size_t>(P) * a.f * 2);
    int32_t* hexp = reinterpret_cast<int32_t*>(base);

    if (!a.x16_ready) {
        cudaError_t e0 = launch_pdl(prep_rows_kernel, dim3((a.T + 7) / 8), dim3(256), 0, s, a.x,
                                    a.T, a.d, x16, xexp);
        trace_mark("decode_prep", s);
        if (e0 != cudaSuccess) return e0;
    }

    Phase up{};
    up.q[0] = a.w1_q; up.q[1] = a.w3_q; up.s[0] = a.w1_s; up.s[1] = a.w3_s;
    up.nmat = 2; up.rows = a.f; up.K = a.d; up.b = x16; up.bexp = xexp; up.b_by_token = 1;
    up.part = upart; up.P = P;
    cudaError_t e = launch_phase<2>(a, up, s, "decode_up");
    if (e != cudaSuccess) return e;

    e = launch_pdl(finish_up_kernel, dim3(P), dim3(kFinishThreads), 0, s,
                   static_cast<const float*>(upart), P, a.f, h16, hexp);
    trace_mark("decode_finish_up", s);
    if (e != cudaSuccess) return e;

    Phase dn{};
    dn.q[0] = a.w2_q; dn.q[1] = a.w2_q; dn.s[0] = a.w2_s; dn.s[1] = a.w2_s;
    dn.nmat = 1; dn.rows = a.d; dn.K = a.f; dn.b = h16; dn.bexp = hexp; dn.b_by_token = 0;
    dn.part = a.y; dn.P = P;
    e = launch_phase<1>(a, dn, s, "decode_down");
    if (e != cudaSuccess) return e;
    return launch_combine(a.y, 2, a.wts, a.inv, a.T, a.k, a.d, a.out, s);
}

}  // namespace k3
