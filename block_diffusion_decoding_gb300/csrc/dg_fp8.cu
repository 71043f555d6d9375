// dg_fp8.cu -- E4M3 (OCP FP8) quantisation of the LM-head operands.
//
// The pages quote their throughput for an FP8 model ("DiffusionGemma Lab",
// section 1; "Parallel Denoising From an Autoregressive Checkpoint", section
// "Finding"); an FP8 weight stream halves the LM head's bytes, which bound
// the step.  A row of n bf16 values x is stored as E4M3 codes with one fp32
// scale: amax = max |x|; if amax == 0 the codes are 0 and the scale 1, else
// inv = fp32(448 / amax), scale = fp32(amax / 448) and
// code_j = E4M3 round-to-nearest-even of fp32(x_j * inv), saturated at +-448;
// the row stands for decode(code_j) * scale.  The hidden states are
// quantised per canvas row, W per vocabulary column (into W8t [V, d]).
#include <cuda_fp8.h>

#include "dg_kernels.h"

namespace dg {

namespace {

DG_DEVICE float bf16_to_f32(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }

DG_DEVICE uint8_t e4m3_code(float v)
{
    return static_cast<uint8_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}

}  // namespace

// One warp per row.
__global__ void __launch_bounds__(256) quantize_rows_e4m3_kernel(const uint16_t *__restrict__ x,
                                                                 int64_t rows, int cols,
                                                                 uint8_t *__restrict__ q,
                                                                 float *__restrict__ scale)
{
    griddep_wait();
    griddep_launch_dependents();
    const int64_t r = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= rows) return;
    const uint16_t *xr = x + r * cols;
    float amax = 0.f;
    for (int j = lane; j < cols; j += 32) amax = fmaxf(amax, fabsf(bf16_to_f32(xr[j])));
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
    uint8_t *qr = q + r * cols;
    if (amax == 0.f) {
        for (int j = lane; j < cols; j += 32) qr[j] = 0;
        if (lane == 0) scale[r] = 1.f;
        return;
    }
    const float inv = __fdiv_rn(448.f, amax);
    if (lane == 0) scale[r] = __fdiv_rn(amax, 448.f);
    for (int j = lane; j < cols; j += 32) qr[j] = e4m3_code(__fmul_rn(bf16_to_f32(xr[j]), inv));
}

// One CTA of 128 threads per row, the row held in registers as 16-byte
// vectors (cols % 8 == 0, cols <= 128 * 8 * kQuantVecs, x 16-byte and q
// 8-byte aligned): one read of x, a block-wide maximum, one write of q.
__global__ void __launch_bounds__(128) quantize_rows_e4m3_vec_kernel(const uint16_t *__restrict__ x,
                                                                     int cols,
                                                                     uint8_t *__restrict__ q,
                                                                     float *__restrict__ scale)
{
    __shared__ float wmax[4];
    griddep_wait();
    griddep_launch_dependents();
    const int64_t r = blockIdx.x;
    const int nv = cols >> 3;
    const uint4 *xr = reinterpret_cast<const uint4 *>(x + r * cols);
    uint4 v[kQuantVecs];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < kQuantVecs; ++i) {
        const int j = static_cast<int>(threadIdx.x) + 128 * i;
        v[i] = j < nv ? __ldg(xr + j) : make_uint4(0, 0, 0, 0);
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            amax = fmaxf(amax, fabsf(bf16_to_f32(static_cast<uint16_t>(w[h] & 0xFFFFu))));
            amax = fmaxf(amax, fabsf(bf16_to_f32(static_cast<uint16_t>(w[h] >> 16))));
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = fmaxf(fmaxf(wmax[0], wmax[1]), fmaxf(wmax[2], wmax[3]));
    const bool zero = amax == 0.f;
    const float inv = zero ? 0.f : __fdiv_rn(448.f, amax);
    if (threadIdx.x == 0) scale[r] = zero ? 1.f : __fdiv_rn(amax, 448.f);
    uint2 *qr = reinterpret_cast<uint2 *>(q + r * cols);
#pragma unroll
    for (int i = 0; i < kQuantVecs; ++i) {
        const int j = static_cast<int>(threadIdx.x) + 128 * i;
        if (j >= nv) break;
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
        uint32_t o[2] = {0u, 0u};
        if (!zero) {
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const uint32_t lo = e4m3_code(__fmul_rn(bf16_to_f32(static_cast<uint16_t>(w[h] & 0xFFFFu)), inv));
                const uint32_t hi = e4m3_code(__fmul_rn(bf16_to_f32(static_cast<uint16_t>(w[h] >> 16)), inv));
                o[h >> 1] |= (lo | (hi << 8)) << (16 * (h & 1));
            }
        }
        qr[j] = make_uint2(o[0], o[1]);
    }
}

// Column maxima of W [d, V] into amax[V]: thread = vocabulary column
// (coalesced along V).
__global__ void __launch_bounds__(256) column_amax_kernel(const uint16_t *__restrict__ w, int d,
                                                         int V, float *__restrict__ amax)
{
    const int v = blockIdx.x * 256 + threadIdx.x;
    if (v >= V) return;
    float m = 0.f;
    for (int k = 0; k < d; ++k) m = fmaxf(m, fabsf(bf16_to_f32(w[static_cast<size_t>(k) * V + v])));
    amax[v] = m;
}

// amax -> scale in place: amax / 448, or 1 for an all-zero column.
__global__ void __launch_bounds__(256) scale_from_amax_kernel(float *__restrict__ s, int n)
{
    const int v = blockIdx.x * 256 + threadIdx.x;
    if (v >= n) return;
    const float m = s[v];
    s[v] = (m > 0.f) ? __fdiv_rn(m, 448.f) : 1.f;
}

// W [d, V] -> W8t [V, d] through 32 x 32 tiles in shared memory, given the
// column maxima.
__global__ void __launch_bounds__(256) quantize_cols_e4m3_kernel(const uint16_t *__restrict__ w,
                                                                 int d, int V,
                                                                 const float *__restrict__ amax,
                                                                 uint8_t *__restrict__ w8t)
{
    __shared__ uint8_t tile[32][33];
    const int v0 = blockIdx.x * 32, k0 = blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 32 x 8
    const int v = v0 + tx;
    float inv = 0.f;
    if (v < V) {
        const float m = amax[v];
        inv = (m > 0.f) ? __fdiv_rn(448.f, m) : 0.f;
    }
    for (int kk = ty; kk < 32; kk += 8) {
        const int k = k0 + kk;
        uint8_t c = 0;
        if (v < V && k < d && inv > 0.f)
            c = e4m3_code(__fmul_rn(bf16_to_f32(w[static_cast<size_t>(k) * V + v]), inv));
        tile[tx][kk] = c;
    }
    __syncthreads();
    for (int vv = ty; vv < 32; vv += 8) {
        const int vo = v0 + vv, ko = k0 + tx;
        if (vo < V && ko < d) w8t[static_cast<size_t>(vo) * d + ko] = tile[vv][tx];
    }
}

// W [d, V] -> the packed LM-head weight [ceil(V / 128)][d][128], zero past
// V: one thread per 16 bytes (8 values; V % 8 == 0, so a chunk is all inside
// or all past V); the 16 chunks of a packed row read one 256-byte stretch of
// a row of W.
__global__ void __launch_bounds__(256) pack_lm_weight_kernel(const uint16_t *__restrict__ w, int d,
                                                             int V, uint16_t *__restrict__ wp)
{
    const int64_t n = static_cast<int64_t>((V + 127) / 128) * d * 16;
    for (int64_t i = blockIdx.x * 256LL + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * 256) {
        const int c8 = static_cast<int>(i & 15);
        const int64_t row = i >> 4;                  // tile * d + k
        const int t = static_cast<int>(row / d), k = static_cast<int>(row % d);
        const int v = t * 128 + c8 * 8;
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (v < V) val = *reinterpret_cast<const uint4 *>(w + static_cast<size_t>(k) * V + v);
        reinterpret_cast<uint4 *>(wp)[i] = val;
    }
}

}  // namespace dg
