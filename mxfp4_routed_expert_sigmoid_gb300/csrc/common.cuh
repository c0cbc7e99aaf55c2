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

}  // namespace k3

// ---------------------------------------------------------------------------
// launchers implemented in the .cu files (host side, return cudaError_t)
// ---------------------------------------------------------------------------
namespace k3 {

// Tracing hook: records an event after a launch when tracing is on (abi.cu).
void trace_mark(const char* name, cudaStream_t s);

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
    // fused permutation outputs (decode path) - may be null
    int32_t* counts;   // [E]
    int32_t* offsets;  // [E+1]
    int32_t* perm;     // [T*k]
    int32_t* inv;      // [T*k]
    int32_t* active;   // [E] ascending experts with count > 0; active[E] = n_active (at index E)
    // optional (decode, latent mode): the router input as f16 rows with one
    // power-of-two exponent per row, written by the last CTA
    uint16_t* x16;     // [T, d_r]
    int32_t* xexp;     // [T]
};

// one warp: row (K bf16) -> f16 * 2^-e with e = floor(log2(max |row|)); returns e
__device__ __forceinline__ int row_to_f16(const uint16_t* src, int K, uint16_t* dst) {
    const int lane = threadIdx.x & 31;
    float amax = 0.0f;
    for (int c = lane * 8; c < K; c += 256) {
        const uint4 v = *reinterpret_cast<const uint4*>(src + c);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[j] << 16)),
                                     fabsf(__uint_as_float(w[j] & 0xFFFF0000u))));
    }
    amax = warp_max(amax);
    const int ex = ilog2f(amax);
    const float sc = exp2i(-ex);
    for (int c = lane * 8; c < K; c += 256) {
        const uint4 v = *reinterpret_cast<const uint4*>(src + c);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint4 o;
        o.x = f32x2_to_f16x2(__uint_as_float(w[0] << 16) * sc, __uint_as_float(w[0] & 0xFFFF0000u) * sc);
        o.y = f32x2_to_f16x2(__uint_as_float(w[1] << 16) * sc, __uint_as_float(w[1] & 0xFFFF0000u) * sc);
        o.z = f32x2_to_f16x2(__uint_as_float(w[2] << 16) * sc, __uint_as_float(w[2] & 0xFFFF0000u) * sc);
        o.w = f32x2_to_f16x2(__uint_as_float(w[3] << 16) * sc, __uint_as_float(w[3] & 0xFFFF0000u) * sc);
        *reinterpret_cast<uint4*>(dst + c) = o;
    }
    return ex;
}

cudaError_t launch_repack(const uint8_t* packed, const uint8_t* scale, int64_t nblocks,
                          uint8_t* out, cudaStream_t s);
cudaError_t launch_unpack(const uint8_t* blocks, int64_t nblocks, uint8_t* packed,
                          uint8_t* scale, cudaStream_t s);

// small T: GEMV logits + (last CTA) top-k [+ permutation if args.counts]
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
cudaError_t launch_permute(const int32_t* idx, int T, int k, int E, int32_t* counts,
                           int32_t* offsets, int32_t* perm, int32_t* inv, int32_t* active,
                           void* scratch, WsHeader* hdr, cudaStream_t s);

cudaError_t launch_rmsnorm(const uint16_t* h, int T, int D, const uint16_t* gamma, float eps,
                           uint16_t* out, cudaStream_t s);

// combine: out[t, :] = bf16(sum_j w[t,j] * (sum_s y[s][inv[t*k+j], :])), j and s in order
cudaError_t launch_combine(const float* y, int nslots, const float* wts, const int32_t* inv, int T,
                           int k, int d, uint16_t* out, cudaStream_t s);

// decode path
struct DecodeArgs {
    const uint8_t *w1_q, *w1_s, *w3_q, *w3_s, *w2_q, *w2_s;
    const uint16_t* x;     // [T, d] bf16 expert input
    int x16_ready;         // 1: the router already wrote the f16 rows into the scratch
    int T, E, k, d, f;
    const int32_t* offsets;  // [E+1]
    const int32_t* perm;     // [T*k]
    const int32_t* active;   // [E+1] list + count at [E]
    const float* wts;        // [T, k]
    const int32_t* inv;      // [T*k]
    void* scratch;           // decode_scratch_bytes(T, k, d, f)
    float* y;                // [2 slots][T*k, d] fp32 partial sums, rows in permuted order
    uint16_t* out;           // [T, d] bf16
    WsHeader* hdr;
    int num_sms;
};
size_t decode_scratch_bytes(int T, int k, int d, int f);
// where the decode scratch keeps the f16 token rows and their exponents
void decode_x16_slots(void* scratch, int T, int d, uint16_t** x16, int32_t** xexp);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);

// grouped (tcgen05) path
struct GroupedArgs {
    const uint8_t *w1_q, *w1_s, *w3_q, *w3_s, *w2_q, *w2_s;
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
                             int out_fp32, WsHeader* hdr, int num_sms, cudaStream_t s);

}  // namespace k3
