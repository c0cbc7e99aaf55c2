// Internal definitions shared by the k3moe CUDA translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/k3moe.h"

namespace k3 {

// ---------------------------------------------------------------------------
// Workspace header (first 256 bytes of every workspace the library uses).
//   status   first device error (k3moe_status), 0 = OK; cleared by get_status
//   info     where the error was raised (kernel-specific code)
//   counters completion tickets of "last CTA finishes the job" kernels; each
//            kernel resets its own counter, so a zero-filled header stays valid
// ---------------------------------------------------------------------------
struct WsHeader {
    int32_t status;
    int32_t info;
    uint32_t counters[30];
    uint32_t pad[32];
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");

enum Counter { CTR_ROUTE = 0, CTR_ROUTE_BIG = 1, CTR_DECODE_B = 2 };

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x, size_t a = kAlign) { return (x + a - 1) / a * a; }

__device__ __forceinline__ void set_error(WsHeader* h, int code, int info) {
    if (atomicCAS(&h->status, 0, code) == 0) h->info = info;
}

// globaltimer in nanoseconds (for bounded waits)
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded waits give up after this long and record K3MOE_ERR_TIMEOUT.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// Device-side kernel timeline (k3moe_trace mode 2).  A stamp area in the
// forward's workspace holds kStampSlots start words then kStampSlots end words;
// the launch that owns slot i records the earliest globaltimer over its CTAs
// at start[i] and the latest at end[i].  A null slot pointer turns it off.
constexpr int kStampSlots = 48;
__device__ __forceinline__ void stamp_start(uint64_t* st) {
    if (st && threadIdx.x == 0) atomicMin(reinterpret_cast<unsigned long long*>(st), global_ns());
}
__device__ __forceinline__ void stamp_end(uint64_t* st) {
    if (st && threadIdx.x == 0) atomicMax(reinterpret_cast<unsigned long long*>(st + kStampSlots), global_ns());
}
// start on construction, end when the scope (and so the CTA's thread 0) exits
struct StampScope {
    uint64_t* st;
    __device__ explicit StampScope(uint64_t* s) : st(s) { stamp_start(st); }
    __device__ ~StampScope() { stamp_end(st); }
};

// ---------------------------------------------------------------------------
// small numeric helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// round-to-nearest-even fp32 -> bf16 bits (finite inputs; NaN stays NaN)
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
    uint32_t u;
    asm("{ .reg .b16 r; cvt.rn.bf16.f32 r, %1; mov.b32 %0, {r, r}; }" : "=r"(u) : "f"(f));
    return static_cast<uint16_t>(u & 0xFFFFu);
}

// 2^n as fp32, exact for every integer n (normal, subnormal, 0 or inf).
__device__ __forceinline__ float exp2i(int n) {
    if (n >= -126 && n <= 127) return __int_as_float((n + 127) << 23);
    return ldexpf(1.0f, n);
}

// Four E2M1 code pairs (one 32-bit word = 8 codes, element 2i in the low
// nibble of byte i) to four f16x2 words with the element order kept: word i
// holds elements 2i (low half) and 2i+1 (high half).
__device__ __forceinline__ void e2m1x8_to_f16x8(uint32_t w, uint32_t& h0, uint32_t& h1,
                                                uint32_t& h2, uint32_t& h3) {
    asm("{\n"
        ".reg .b8 b0, b1, b2, b3;\n"
        "mov.b32 {b0, b1, b2, b3}, %4;\n"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n"
        "}"
        : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
        : "r"(w));
}

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ float2 f16x2_to_f32x2(uint32_t h) {
    float2 r;
    asm("{ .reg .f16 lo, hi; mov.b32 {lo, hi}, %2; cvt.f32.f16 %0, lo; cvt.f32.f16 %1, hi; }"
        : "=f"(r.x), "=f"(r.y)
        : "r"(h));
    return r;
}

// pack two fp32 into f16x2 (round to nearest even); a -> low half
__device__ __forceinline__ uint32_t f32x2_to_f16x2(float a, float b) {
    uint32_t d;
    asm("cvt.rn.f16x2.f32 %0, %2, %1;" : "=r"(d) : "f"(a), "f"(b));
    return d;
}

// floor(log2(|x|)) for finite nonzero x (exact, from the exponent field);
// 0 for x == 0.
__device__ __forceinline__ int ilog2f(float x) {
    if (x == 0.0f) return 0;
    int e;
    frexpf(x, &e);  // x = m * 2^e, 0.5 <= |m| < 1
    return e - 1;
}

// v * 2^n without a branch, for use inside unrolled loops: n is clamped to
// [-252, 254] and applied as two power-of-two factors 2^hi * 2^lo, both
// normal floats (hi in [-126, 127]); exact except that a result below the
// normal range may round twice.
__device__ __forceinline__ float mul_pow2(float v, int n) {
    n = max(min(n, 254), -252);
    const int lo = n < -126 ? n + 126 : (n > 127 ? n - 127 : 0);
    const int hi = n - lo;
    return v * __int_as_float((hi + 127) << 23) * __int_as_float((lo + 127) << 23);
}

// f16 bit pattern of 2^n for n in [-24, 15]; 0 below (flush), inf above.
__device__ __forceinline__ uint16_t f16_pow2(int n) {
    if (n < -24) return 0;
    if (n < -14) return static_cast<uint16_t>(1u << (n + 24));
    if (n > 15) return 0x7C00;
    return static_cast<uint16_t>((n + 15) << 10);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Programmatic dependent launch.  A kernel launched with launch_pdl() may
// start while its predecessor on the stream is still running: it must call
// pdl_wait() before it touches anything the predecessor writes or reads.
// pdl_trigger() lets the next kernel begin launching early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// ---------------------------------------------------------------------------
// Activations for the block-scaled tensor-core path: every 32-element block
// of a row is written as kTerms E2M1 codes per element, each term with its
// own E8M0 block scale, so that v ~= sum_j e2m1(q_j) * 2^(s_j - 127).  Term
// j + 1 encodes what term j left over (exactly: the remainder of a
// round-to-nearest is representable), so each term adds about 3.3 bits; five
// terms put the layer output within about 1e-4 of its RMS.
// ---------------------------------------------------------------------------
constexpr int kTerms = 5;

// Smallest e >= -127 with amax * 2^-e <= 6 (the largest E2M1 magnitude), from
// the exponent and mantissa fields: amax = (1 + m) 2^E fits at e = E - 2 iff
// 1 + m <= 1.5.  The E8M0 byte is e + 127, so e stays at -127 or above (byte
// 255 is NaN): zero, subnormal and lowest-binade amax (below 2^-125) give
// -127, where amax * 2^127 < 4 still fits.
__device__ __forceinline__ int e2m1_scale_exp(float amax) {
    const uint32_t u = __float_as_uint(amax);
    const int ef = static_cast<int>((u >> 23) & 0xFFu);
    const int e = ef - 127 - 2 + ((u & 0x7FFFFFu) > 0x400000u ? 1 : 0);
    return e < -127 ? -127 : e;
}

// fp32 -> E2M1 code (round to nearest even, saturating to +-6), low 4 bits
__device__ __forceinline__ uint32_t e2m1_code(float v) {
    uint32_t r;
    asm("{ .reg .b8 c; cvt.rn.satfinite.e2m1x2.f32 c, %1, %1; mov.b32 %0, {c, c, c, c}; }" : "=r"(r) : "f"(v));
    return r & 0xFu;
}

// E2M1 code -> fp32 (exact)
__device__ __forceinline__ float e2m1_float(uint32_t code) {
    uint32_t h;
    asm("{ .reg .b8 c0, c1, c2, c3; mov.b32 {c0, c1, c2, c3}, %1; cvt.rn.f16x2.e2m1x2 %0, c0; }"
        : "=r"(h)
        : "r"(code));
    return f16x2_to_f32x2(h).x;
}

// One 32-element block held by a warp (lane = element) -> kTerms codes of
// this lane's element and the kTerms scale bytes (warp-uniform).
__device__ __forceinline__ void quantize_terms(float v, uint32_t (&q)[kTerms], uint32_t (&sb)[kTerms]) {
    float res = v;
#pragma unroll
    for (int j = 0; j < kTerms; ++j) {
        // largest |res| of the block: non-negative floats order like their bits
        const float amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(res))));
        const int e = e2m1_scale_exp(amax);
        q[j] = e2m1_code(res * exp2i(-e));
        sb[j] = static_cast<uint32_t>(e + 127);
        res = res - e2m1_float(q[j]) * exp2i(e);
    }
}

// Two fp32 values -> one byte of E2M1 codes (lo in the low nibble; round to
// nearest even, saturating), and the byte back to the two exact values.
__device__ __forceinline__ uint32_t e2m1x2_code(float lo, float hi) {
    uint32_t r;
    asm("{ .reg .b8 c; cvt.rn.satfinite.e2m1x2.f32 c, %1, %2; mov.b32 %0, {c, c, c, c}; }"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return r & 0xFFu;
}
__device__ __forceinline__ float2 e2m1x2_float(uint32_t byte) {
    uint32_t h;
    asm("{ .reg .b8 c0, c1, c2, c3; mov.b32 {c0, c1, c2, c3}, %1; cvt.rn.f16x2.e2m1x2 %0, c0; }"
        : "=r"(h)
        : "r"(byte));
    return f16x2_to_f32x2(h);
}

// The same terms with 8 consecutive elements per lane: lanes 4m .. 4m + 3 hold
// one 32-element block (lane 4m + r elements 8r .. 8r + 7), so a term's block
// maximum takes two shuffles and its codes pack into one word per lane
// (element 8r + i in nibble i).  v is left holding the residual.
template <int TERMS>
__device__ __forceinline__ void quantize8_terms(float (&v)[8], uint32_t (&w)[TERMS], uint32_t (&sb)[TERMS]) {
#pragma unroll
    for (int j = 0; j < TERMS; ++j) {
        float m = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        const int e = e2m1_scale_exp(m);
        const float inv = exp2i(-e), sc = exp2i(e);
        uint32_t word = 0;
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
            const uint32_t byte = e2m1x2_code(v[i] * inv, v[i + 1] * inv);
            const float2 d = e2m1x2_float(byte);
            v[i] = fmaf(-d.x, sc, v[i]);
            v[i + 1] = fmaf(-d.y, sc, v[i + 1]);
            word |= byte << (4 * i);
        }
        w[j] = word;
        sb[j] = static_cast<uint32_t>(e + 127);
    }
}

// B operand layout of the block-scaled MMA (kind::mxf4: packed E2M1, two
// codes per byte, element 2i in the low nibble), per 256-wide K chunk:
//   codes : N rows x 128 bytes, row n = kTerms * token + term, stored with the
//           128-byte swizzle of the tensor-core K-major layout (16-byte chunk
//           c of row n at chunk c ^ (n % 8); a 32-element block is exactly one
//           16-byte chunk), so one bulk copy lands it ready for the MMA;
//   scales: per 128-wide K group a 512-byte atom, byte 16 (n % 32) + 4 (n / 32)
//           + kb for row n and 32-block kb of the group (the layout tcgen05.cp
//           32x128b.warpx4 spreads over the TMEM lanes the MMA reads).
__device__ __forceinline__ uint32_t sf_atom_offset(int n, int kb) {
    return static_cast<uint32_t>(16 * (n & 31) + 4 * (n >> 5) + kb);
}

// Writes the quantised block (warp, lane = element) of token t into the B
// layout: 32-block kb (0..7) of the 256-wide chunk whose codes start at
// `codes`; `scales` is the atom of the chunk's first 128-wide group (the
// second follows 512 bytes later).  Lane pairs share a byte, lanes 8i..8i+7
// one 32-bit store.
__device__ __forceinline__ void store_terms(const uint32_t (&q)[kTerms], const uint32_t (&sb)[kTerms],
                                            int t, int kb, uint8_t* codes, uint8_t* scales) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int j = 0; j < kTerms; ++j) {
        const uint32_t b = q[j] | (__shfl_down_sync(0xffffffffu, q[j], 1) << 4);   // even lanes
        uint32_t w = b;
        w |= __shfl_down_sync(0xffffffffu, b, 2) << 8;
        w |= __shfl_down_sync(0xffffffffu, b, 4) << 16;
        w |= __shfl_down_sync(0xffffffffu, b, 6) << 24;
        const int n = kTerms * t + j;
        if ((lane & 7) == 0)
            *reinterpret_cast<uint32_t*>(codes + n * 128 + (((kb ^ (n & 7)) & 7) << 4) + (lane >> 1)) = w;
        if (lane == 0) scales[(kb >> 2) * 512 + sf_atom_offset(n, kb & 3)] = static_cast<uint8_t>(sb[j]);
    }
}

}  // namespace k3

// ---------------------------------------------------------------------------
// launchers implemented in the .cu files (host side, return cudaError_t)
// ---------------------------------------------------------------------------
namespace k3 {

// Tracing hooks (abi.cu): trace_mark records an event after a launch when
// event tracing is on; trace_stamp, called before a launch, returns the
// launch's stamp slot when device stamps are on inside a forward (else null).
void trace_mark(const char* name, cudaStream_t s);
uint64_t* trace_stamp(const char* name);

// Kernel launch with programmatic stream serialisation (see pdl_wait).
bool pdl_enabled();
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

struct RouteArgs {
    const uint16_t* x;
    int T, d_r;
    const uint16_t* w;
    const float* bias;
    int E, k;
    int32_t* idx;
    float* wts;
    float* logits;     // [T, E] fp32 (always written; in the workspace if the caller passes none)
    WsHeader* hdr;
    // decode: the ascending experts that received any token, count at [E]
    // (written by the small-T top-k kernel; null = not wanted)
    int32_t* active;   // [E + 1]
    // optional (decode, latent mode): the router input quantised for the
    // block-scaled expert kernels (codes [d_r / 256][xq_n][128], scale atoms
    // [d_r / 128][512]); the CTAs share the work
    uint8_t* xq;
    uint8_t* xsf;
    int xq_n;          // MMA N: rows per stage (>= kTerms * T)
    uint64_t* st_a;    // stamp slots: logits kernel, top-k kernel (null: off)
    uint64_t* st_b;
};

cudaError_t launch_repack(const uint8_t* packed, const uint8_t* scale, int64_t nblocks,
                          uint8_t* out, cudaStream_t s);
cudaError_t launch_unpack(const uint8_t* blocks, int64_t nblocks, uint8_t* packed,
                          uint8_t* scale, cudaStream_t s);

// small T: GEMV logits (+ E2M1 terms of the rows if a.xq), then the top-k
// kernel (+ active expert list if a.active)
cudaError_t launch_route_small(const RouteArgs& a, cudaStream_t s);
// the same with library-owned static scratch (no caller workspace)
constexpr int kNoAllocMaxT = 8;
constexpr int kNoAllocMaxE = 1024;
cudaError_t launch_route_noalloc(RouteArgs a, cudaStream_t s);
// any T: logits already in a.logits -> top-k
cudaError_t launch_topk(const RouteArgs& a, cudaStream_t s);
// SIMT GEMV/GEMM logits for moderate T (no top-k)
cudaError_t launch_logits_simt(const RouteArgs& a, cudaStream_t s);
// permutation of any T (chunked, deterministic); scratch >= permute_scratch_bytes
size_t permute_scratch_bytes(int T, int E);
// clamp = 1: idx is library-owned scratch; an entry outside [0, E) is recorded
// and rewritten to 0 (else it is recorded and left out of the permutation)
cudaError_t launch_permute(const int32_t* idx, int T, int k, int E, int32_t* counts,
                           int32_t* offsets, int32_t* perm, int32_t* inv, int32_t* active,
                           void* scratch, WsHeader* hdr, cudaStream_t s, int clamp = 0);

cudaError_t launch_rmsnorm(const uint16_t* h, int T, int D, const uint16_t* gamma, float eps,
                           uint16_t* out, cudaStream_t s);

// combine: out[t, :] = bf16(sum_j w[t,j] * (sum_s y[s][inv[t*k+j], :])), j and s in order
cudaError_t launch_combine(const float* y, int nslots, const float* wts, const int32_t* inv, int T,
                           int k, int d, uint16_t* out, cudaStream_t s);


// block-scaled tensor-core decode path (mx.cu)
struct MxDecodeArgs {
    const uint8_t *w1_q, *w3_q, *w2_q;  // E2M1 codes
    const uint8_t *w1_sf, *w3_sf, *w2_sf;  // E8M0 scales: prepared atoms, or canonical rows (sf_canon)
    int sf_canon;             // 1: w*_sf are the canonical [rows, K / 32] arrays (d, f multiples of 512)
    const uint16_t* x;        // [T, d] bf16 expert input (read when !xq_ready)
    int xq_ready;             // 1: the router already wrote the E2M1 terms
    int T, E, k, d, f;
    const int32_t* active;    // [E + 1] active experts ascending, count at [E]
    const int32_t* slot_of;   // expert -> weight slot of the w arrays (null: the expert itself)
    int nslots;               // expert slots the w arrays hold (E without a cache)
    int ggml;                 // 1: w*_q hold ggml 17-byte blocks (w*_sf unused)
    const int32_t* idx;       // [T, k]
    const float* wts;         // [T, k]
    void* scratch;            // mx_decode_scratch_bytes(T, E, k, d, f)
    uint16_t* out;            // [T, d] bf16
    WsHeader* hdr;
    int num_sms;
    int inject;               // test aid (k3moe_inject_fault) for the up pass
};
size_t mx_decode_scratch_bytes(int T, int E, int k, int d, int f);
// where the decode scratch keeps the quantised token rows (router output)
void mx_decode_xq_slots(void* scratch, int T, int E, int k, int d, int f, uint8_t** xq, uint8_t** xsf,
                        int* N);
cudaError_t launch_mx_decode(const MxDecodeArgs& a, cudaStream_t s);
// unit-grouped streaming forward (more tokens, few per expert): the experts'
// sorted token lists (from the permutation) are cut into units of at most 16
// tokens and streamed like the decode path
struct MxUnitsArgs {
    const uint8_t *w1_q, *w3_q, *w2_q;     // E2M1 codes
    const uint8_t *w1_sf, *w3_sf, *w2_sf;  // E8M0 scales: prepared atoms, or canonical rows (sf_canon)
    int sf_canon;             // 1: w*_sf are the canonical [rows, K / 32] arrays (d, f multiples of 512)
    const uint16_t* x;        // [T, d] bf16 expert input
    int T, E, k, d, f;
    const int32_t* counts;    // [E]
    const int32_t* offsets;   // [E + 1]
    const int32_t* perm;      // [T k] sorted row -> (token, slot) pair
    const int32_t* inv;       // [T k] pair -> sorted row
    const int32_t* idx;       // [T, k]
    const float* wts;         // [T, k]
    const int32_t* slot_of;   // expert -> weight slot (null: the expert itself)
    int nslots;               // expert slots the w arrays hold (E without a cache)
    int ggml;                 // 1: w*_q hold ggml 17-byte blocks (w*_sf unused)
    void* scratch;            // mx_units_scratch_bytes(T, E, k, d, f)
    uint16_t* out;            // [T, d] bf16
    WsHeader* hdr;
    int num_sms;
    int inject;               // test aid (k3moe_inject_fault) for the up pass
};
size_t mx_units_scratch_bytes(int T, int E, int k, int d, int f);
cudaError_t launch_mx_units(const MxUnitsArgs& a, cudaStream_t s);
// device expert cache (cache.cu).  The caller's state buffer holds a 256-byte
// header, then slot_of [E], expert_of [S], stamp [S], miss_e [S], miss_slot [S]
// (int32 / uint32, each array 256-byte aligned).
constexpr uint32_t kCacheMagic = 0x4b33c4c1u;
struct CacheHeader {
    uint32_t magic;         // kCacheMagic after k3moe_cache_init
    int32_t E, slots;
    uint32_t clock;         // calls served; a slot's stamp is the clock of its last use
    int32_t last_miss, last_hit;
    int32_t pad0[2];
    unsigned long long calls, hits, misses, bytes;  // totals since init
    uint32_t pad[48];
};
static_assert(sizeof(CacheHeader) == 256, "cache header is 256 bytes");
struct CacheView {
    CacheHeader* h;
    int32_t* slot_of;    // [E] slot holding the expert, -1 = not resident; right after the header
    int32_t* expert_of;  // [S] expert in the slot, -1 = empty
    uint32_t* stamp;     // [S] clock of the slot's last use (0 = never)
    int32_t* miss_e;     // [S] experts to fetch in this call, ascending
    int32_t* miss_slot;  // [S] the slot each of them goes to
};
size_t cache_state_bytes(int E, int slots);
CacheView cache_view(void* state, int E, int slots);
// where the fetched bytes come from (device addresses of host-resident
// arrays) and go to (the slot arrays); per expert and matrix q_bytes of
// codes and sf_bytes of prepared scale atoms, in the order w1, w3, w2
struct CacheFillArgs {
    const uint8_t* src_q[3];
    const uint8_t* src_sf[3];
    uint8_t* dst_q[3];
    uint8_t* dst_sf[3];
    size_t q_bytes, sf_bytes;
};
cudaError_t launch_cache_init(void* state, int E, int slots, cudaStream_t s);
// after the active list is final: slot assignment (one CTA), then the copy of
// the missing experts into their slots (all SMs)
cudaError_t launch_cache_update(void* state, int E, int slots, const int32_t* active,
                                const CacheFillArgs& f, WsHeader* hdr, int num_sms, cudaStream_t s);

// canonical E8M0 scales [E, R, K/32] <-> prepared atoms (inverse = 1: atoms -> canonical); the
// atoms of an expert fill ceil(R / 128) x ceil(K / 128) atoms of 512 bytes (zero padding)
size_t prepared_sf_bytes(int64_t E, int R, int K);
cudaError_t launch_prepare_sf(const uint8_t* canon, int64_t E, int R, int K, uint8_t* atoms, int inverse,
                              cudaStream_t s);

// grouped (tcgen05) path
struct GroupedArgs {
    const uint8_t *w1_q, *w3_q, *w2_q;  // E2M1 codes
    const uint8_t *w1_sf, *w3_sf, *w2_sf;  // E8M0 scales: prepared atoms, or canonical rows (sf_canon)
    int sf_canon;            // 1: w*_sf are the canonical [rows, K / 32] arrays (d, f multiples of 512)
    const uint16_t* x;       // [T, d] bf16 expert input
    int T, E, k, d, f;
    const int32_t* counts;   // [E]
    const int32_t* offsets;  // [E+1]
    const int32_t* perm;     // [T*k]
    const int32_t* inv;      // [T*k]
    const float* wts;        // [T, k]
    uint16_t* xp;            // [T*k, d] f16 prescaled rows (permuted order)
    int32_t* xp_exp;         // [T*k]
    float* hf;               // [T*k, f] fp32 (up epilogue output)
    uint32_t* h_amax;        // [T*k] fp32 bits of max |h| per row
    uint16_t* hp;            // [T*k, f] f16 prescaled h
    int32_t* hp_exp;         // [T*k]
    float* y;                // [T*k, d] fp32
    int32_t* tiles;          // two tile lists (up, down), tiles_cap + 1 int4 entries each
    int tiles_cap;
    uint16_t* out;           // [T, d] bf16
    WsHeader* hdr;
    int num_sms;
};
size_t grouped_tile_cap(int T, int E, int k, int d, int f);
cudaError_t launch_grouped(const GroupedArgs& a, cudaStream_t s);

// dense bf16 GEMM (tcgen05): out[t, n] = sum_c x[t, c] w[n, c]
cudaError_t launch_gemm_bf16(const uint16_t* x, const uint16_t* w, int T, int N, int K, void* out,
                             int out_fp32, WsHeader* hdr, int num_sms, cudaStream_t s,
                             const char* name = "gemm_bf16");

}  // namespace k3
