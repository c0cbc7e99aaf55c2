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

__device__ __forceinline__ int max4_bytes(uint32_t w) {
    const int a = max(static_cast<int>(w & 0xFF), static_cast<int>((w >> 8) & 0xFF));
    const int b = max(static_cast<int>((w >> 16) & 0xFF), static_cast<int>(w >> 24));
    return max(a, b);
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

struct Stage {
    uint4 w[2][2];    // [matrix][row g / row g + 8]
    uint32_t s[2][2]; // scale words
    uint4 x[4];       // 32 f16 of the token block
};

__device__ __forceinline__ void load_stage(const Phase& ph, Stage& st, size_t wrow0, size_t wrow8,
                                           int c, int t, const uint16_t* brow, bool has_tok) {
    const int blk = 4 * c + t;
    const int nb = ph.K / 32;
    const bool blk_ok = blk < nb;
    const size_t kq = static_cast<size_t>(ph.K / 2), ks = static_cast<size_t>(nb);
#pragma unroll
    for (int m = 0; m < 2; ++m) {
        if (m < ph.nmat) {
            st.w[m][0] = blk_ok ? ldg_nc_v4(ph.q[m] + wrow0 * kq + 16 * blk) : make_uint4(0, 0, 0, 0);
            st.w[m][1] = blk_ok ? ldg_nc_v4(ph.q[m] + wrow8 * kq + 16 * blk) : make_uint4(0, 0, 0, 0);
            const uint8_t* s0 = ph.s[m] + wrow0 * ks + 4 * c;
            const uint8_t* s8 = ph.s[m] + wrow8 * ks + 4 * c;
            if ((nb & 3) == 0) {
                // rows of the scale array are 4-byte aligned: one word = blocks 4c..4c+3
                st.s[m][0] = __ldg(reinterpret_cast<const uint32_t*>(s0));
                st.s[m][1] = __ldg(reinterpret_cast<const uint32_t*>(s8));
            } else {
                uint32_t v0 = 0, v8 = 0;
                for (int b = 0; b < 4; ++b) {
                    if (4 * c + b < nb) {
                        v0 |= static_cast<uint32_t>(__ldg(s0 + b)) << (8 * b);
                        v8 |= static_cast<uint32_t>(__ldg(s8 + b)) << (8 * b);
                    }
                }
                st.s[m][0] = v0;
                st.s[m][1] = v8;
            }
        }
    }
    if (has_tok && blk_ok) {
        const uint4* xb = reinterpret_cast<const uint4*>(brow + 32 * blk);
#pragma unroll
        for (int i = 0; i < 4; ++i) st.x[i] = xb[i];
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) st.x[i] = make_uint4(0, 0, 0, 0);
    }
}

template <int NMAT>
__device__ __forceinline__ void compute_stage(const Stage& st, int t, float (&tot)[NMAT][4]) {
    const uint32_t xw[16] = {st.x[0].x, st.x[0].y, st.x[0].z, st.x[0].w, st.x[1].x, st.x[1].y,
                             st.x[1].z, st.x[1].w, st.x[2].x, st.x[2].y, st.x[2].z, st.x[2].w,
                             st.x[3].x, st.x[3].y, st.x[3].z, st.x[3].w};
#pragma unroll
    for (int m = 0; m < NMAT; ++m) {
        const int eb0 = (st.s[m][0] >> (8 * t)) & 0xFF, eb8 = (st.s[m][1] >> (8 * t)) & 0xFF;
        const int er0 = max4_bytes(st.s[m][0]), er8 = max4_bytes(st.s[m][1]);
        const uint32_t h0 = f16_pow2(eb0 - er0), h8 = f16_pow2(eb8 - er8);
        uint32_t w0[16], w8[16];
        convert_scaled(st.w[m][0], h0 | (h0 << 16), w0);
        convert_scaled(st.w[m][1], h8 | (h8 << 16), w8);
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
}

// Stream-K phase: partial sums of (selected expert, 16-row tile) over each warp's
// share of the K chunks.
template <int NMAT>
__global__ void __launch_bounds__(kThreads)
decode_phase_kernel(DecodeArgs a, Phase ph) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int64_t warp = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;
    const int U = a.active[a.E];
    const int R = ph.rows / 16;
    const int C = (ph.K + 127) / 128;
    const int64_t n_tiles = static_cast<int64_t>(U) * R;
    const int64_t W = n_tiles * C;
    const int64_t G = nwarps < n_tiles ? nwarps : n_tiles;  // each range >= one tile
    if (warp >= G) return;
    const int64_t start = W * warp / G, end = W * (warp + 1) / G;
    for (int64_t u = start; u < end;) {
        const int64_t tile = u / C;
        const int c0 = static_cast<int>(u - tile * C);
        const int64_t left = end - tile * C;
        const int c1 = left < C ? static_cast<int>(left) : C;
        const int au = static_cast<int>(tile / R), rt = static_cast<int>(tile % R);
        const int e = a.active[au];
        const int o0 = a.offsets[e];
        const int n = min(a.offsets[e + 1] - o0, kMaxTok);
        const bool has_tok = g < n;
        const int brow_idx = has_tok ? (ph.b_by_token ? a.perm[o0 + g] / a.k : o0 + g) : 0;
        const uint16_t* brow = ph.b + static_cast<size_t>(brow_idx) * ph.K;
        const size_t wrow0 = static_cast<size_t>(e) * ph.rows + rt * 16 + g;
        const size_t wrow8 = wrow0 + 8;
        float tot[NMAT][4];
#pragma unroll
        for (int m = 0; m < NMAT; ++m) tot[m][0] = tot[m][1] = tot[m][2] = tot[m][3] = 0.0f;
        // two-deep software pipeline over the chunks (stages named statically so
        // they stay in registers)
        Stage sa, sb;
        load_stage(ph, sa, wrow0, wrow8, c0, t, brow, has_tok);
        for (int c = c0; c < c1; c += 2) {
            if (c + 1 < c1) load_stage(ph, sb, wrow0, wrow8, c + 1, t, brow, has_tok);
            compute_stage<NMAT>(sa, t, tot);
            if (c + 1 < c1) {
                if (c + 2 < c1) load_stage(ph, sa, wrow0, wrow8, c + 2, t, brow, has_tok);
                compute_stage<NMAT>(sb, t, tot);
            }
        }
        // write the partial sums of tokens 2t, 2t+1 (rows g, g+8)
        const int slot = c0 == 0 ? 0 : 1;
        const bool whole = c0 == 0 && c1 == C;
        const int r0 = rt * 16 + g;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int tok = 2 * t + q;
            if (tok >= n) continue;
            const int pr = o0 + tok;
            const int bi = ph.b_by_token ? a.perm[pr] / a.k : pr;
            const float sx = exp2i(ph.bexp[bi]);
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
        u = tile * C + c1;
    }
}

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
// per-row exponent.  One warp per pair row; pairs beyond the selection skip.
__global__ void __launch_bounds__(256)
finish_up_kernel(const float* __restrict__ part, int P, int f, uint16_t* __restrict__ h16,
                 int32_t* __restrict__ hexp) {
    pdl_wait();
    pdl_trigger();
    const int p = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (p >= P) return;
    const size_t plane = static_cast<size_t>(P) * f;
    const float* g0 = part + static_cast<size_t>(p) * f;
    const float* g1 = g0 + plane;
    const float* u0 = g0 + 2 * plane;
    const float* u1 = g0 + 3 * plane;
    float amax = 0.0f;
    for (int c = lane * 4; c < f; c += 128) {
        const float4 a0 = *reinterpret_cast<const float4*>(g0 + c), a1 = *reinterpret_cast<const float4*>(g1 + c);
        const float4 b0 = *reinterpret_cast<const float4*>(u0 + c), b1 = *reinterpret_cast<const float4*>(u1 + c);
        amax = fmaxf(amax, fabsf(silu_f32(a0.x + a1.x) * (b0.x + b1.x)));
        amax = fmaxf(amax, fabsf(silu_f32(a0.y + a1.y) * (b0.y + b1.y)));
        amax = fmaxf(amax, fabsf(silu_f32(a0.z + a1.z) * (b0.z + b1.z)));
        amax = fmaxf(amax, fabsf(silu_f32(a0.w + a1.w) * (b0.w + b1.w)));
    }
    amax = warp_max(amax);
    const int ex = ilog2f(amax);
    const float sc = exp2i(-ex);
    uint16_t* dst = h16 + static_cast<size_t>(p) * f;
    for (int c = lane * 4; c < f; c += 128) {
        const float4 a0 = *reinterpret_cast<const float4*>(g0 + c), a1 = *reinterpret_cast<const float4*>(g1 + c);
        const float4 b0 = *reinterpret_cast<const float4*>(u0 + c), b1 = *reinterpret_cast<const float4*>(u1 + c);
        uint2 o;
        o.x = f32x2_to_f16x2(silu_f32(a0.x + a1.x) * (b0.x + b1.x) * sc,
                             silu_f32(a0.y + a1.y) * (b0.y + b1.y) * sc);
        o.y = f32x2_to_f16x2(silu_f32(a0.z + a1.z) * (b0.z + b1.z) * sc,
                             silu_f32(a0.w + a1.w) * (b0.w + b1.w) * sc);
        *reinterpret_cast<uint2*>(dst + c) = o;
    }
    if (lane == 0) hexp[p] = ex;
}

template <int NMAT>
cudaError_t launch_phase(const DecodeArgs& a, const Phase& ph, cudaStream_t s, const char* name) {
    // four CTAs of four warps per SM; the kernel trims the warp count so that
    // every warp owns at least one whole tile of K chunks
    const int grid = 4 * a.num_sms;
    const cudaError_t e = launch_pdl(decode_phase_kernel<NMAT>, dim3(grid), dim3(kThreads), 0, s, a, ph);
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

    e = launch_pdl(finish_up_kernel, dim3((P + 7) / 8), dim3(256), 0, s,
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
