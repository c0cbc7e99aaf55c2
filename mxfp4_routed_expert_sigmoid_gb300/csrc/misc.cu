// RMSNorm of the latent block and the deterministic weighted combine.
//
// RMSNorm (the ffn_routed_norm tensor of llama.cpp PR #26185 "model: add
// Kimi-K3 text model", review by GrEarl, section "Dry run"; epsilon 1e-5 from
// Lucebox PR #573, section "DSpark acceptance-contract correction"):
//   out = bf16(h * (1 / sqrt(mean(h^2) + eps)) * gamma), fp32 arithmetic,
//   one CTA per row, the sum of squares reduced in a fixed tree order.
//
// Combine: out[t, :] = bf16(sum_j w[t, j] * y[inv[t*k + j], :]), the k terms
// added in slot order j = 0..k-1 in fp32, so the result does not depend on
// how the expert rows were scheduled.
#include "common.cuh"

namespace k3 {
namespace {

constexpr int kNormThreads = 256;

__global__ void __launch_bounds__(kNormThreads)
rmsnorm_kernel(const uint16_t* __restrict__ h, int D, const uint16_t* __restrict__ gamma,
               float eps, uint16_t* __restrict__ out, uint64_t* st) {
    StampScope stamp(st);
    __shared__ float part[kNormThreads / 32];
    __shared__ float inv_rms_s;
    const size_t row = blockIdx.x;
    const uint16_t* src = h + row * D;
    const int nvec = D / 8;
    float ss = 0.0f;
    for (int v = threadIdx.x; v < nvec; v += kNormThreads) {
        const uint4 w = *reinterpret_cast<const uint4*>(src + 8 * v);
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float a = __uint_as_float(ww[j] << 16), b = __uint_as_float(ww[j] & 0xFFFF0000u);
            ss = fmaf(a, a, ss);
            ss = fmaf(b, b, ss);
        }
    }
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.0f;
        for (int w = 0; w < kNormThreads / 32; ++w) t += part[w];
        inv_rms_s = 1.0f / sqrtf(t / static_cast<float>(D) + eps);
    }
    __syncthreads();
    const float r = inv_rms_s;
    uint16_t* dst = out + row * D;
    for (int v = threadIdx.x; v < nvec; v += kNormThreads) {
        const uint4 w = *reinterpret_cast<const uint4*>(src + 8 * v);
        const uint4 g = *reinterpret_cast<const uint4*>(gamma + 8 * v);
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
        const uint32_t gg[4] = {g.x, g.y, g.z, g.w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float a = __uint_as_float(ww[j] << 16) * r * __uint_as_float(gg[j] << 16);
            const float b = __uint_as_float(ww[j] & 0xFFFF0000u) * r * __uint_as_float(gg[j] & 0xFFFF0000u);
            o[j] = static_cast<uint32_t>(f32_to_bf16(a)) | (static_cast<uint32_t>(f32_to_bf16(b)) << 16);
        }
        *reinterpret_cast<uint4*>(dst + 8 * v) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// 128 threads x 4 columns per CTA; grid (ceil(d / 512), T).  The token's k
// (row, weight) pairs are staged in shared memory first, so the loads of the
// k rows are independent and issue together.
constexpr int kCombineThreads = 128;

__global__ void __launch_bounds__(kCombineThreads)
combine_kernel(const float* __restrict__ y, int nslots, size_t slot_stride,
               const float* __restrict__ wts, const int32_t* __restrict__ inv, int k, int d,
               uint16_t* __restrict__ out, uint64_t* st) {
    __shared__ int rows[32];
    __shared__ float wk[32];
    pdl_wait();
    pdl_trigger();
    StampScope stamp(st);
    const int t = blockIdx.y;
    if (threadIdx.x < k) {
        rows[threadIdx.x] = inv[t * k + threadIdx.x];
        wk[threadIdx.x] = wts[t * k + threadIdx.x];
    }
    __syncthreads();
    const int c = (blockIdx.x * kCombineThreads + threadIdx.x) * 4;
    if (c >= d) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int j = 0; j < k; ++j) {
        const float* yr = y + static_cast<size_t>(rows[j]) * d + c;
        float4 v = *reinterpret_cast<const float4*>(yr);
        if (nslots > 1) {
            const float4 v2 = *reinterpret_cast<const float4*>(yr + slot_stride);
            v.x += v2.x; v.y += v2.y; v.z += v2.z; v.w += v2.w;
        }
        const float w = wk[j];
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
    }
    uint2 o;
    o.x = static_cast<uint32_t>(f32_to_bf16(acc.x)) | (static_cast<uint32_t>(f32_to_bf16(acc.y)) << 16);
    o.y = static_cast<uint32_t>(f32_to_bf16(acc.z)) | (static_cast<uint32_t>(f32_to_bf16(acc.w)) << 16);
    *reinterpret_cast<uint2*>(out + static_cast<size_t>(t) * d + c) = o;
}

}  // namespace

cudaError_t launch_rmsnorm(const uint16_t* h, int T, int D, const uint16_t* gamma, float eps,
                           uint16_t* out, cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    rmsnorm_kernel<<<T, kNormThreads, 0, s>>>(h, D, gamma, eps, out, trace_stamp("rmsnorm"));
    trace_mark("rmsnorm", s);
    return cudaGetLastError();
}

cudaError_t launch_combine(const float* y, int nslots, const float* wts, const int32_t* inv, int T,
                           int k, int d, uint16_t* out, cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    dim3 grid((d + 4 * kCombineThreads - 1) / (4 * kCombineThreads), T);
    const size_t slot_stride = static_cast<size_t>(T) * k * d;
    const cudaError_t e = launch_pdl(combine_kernel, grid, dim3(kCombineThreads), 0, s, y, nslots, slot_stride,
                                     wts, inv, k, d, out, trace_stamp("combine"));
    trace_mark("combine", s);
    return e;
}

}  // namespace k3
