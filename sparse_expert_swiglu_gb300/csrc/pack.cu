// INT2 quantisation of W^up and its inverse storage step.
//
// FloE ("FloE: On-the-Fly MoE Inference on Memory-constrained GPU", sec. 三
// "混合压缩策略") stores the up projection as INT2 (Q(.)); the scheme itself is
// not given on the page.  The one implemented here is asymmetric min/max per
// (64-row group, column) with fp16 scale and zero point, every step in fp32 IEEE
// arithmetic so that it is reproducible bit for bit:
//   scale = fp16((max - min) / 3)  (1 if that rounds to 0)
//   zero  = fp16(clamp(-min / scale, +-65504))
//   q     = clamp(rint(w / scale + zero), 0, 3)
#include "common.cuh"

namespace sesg {

// One thread per (column j, group g): scale and zero into the block's (scale, zero) table.
__global__ void pack_scale_zero_kernel(const __half* __restrict__ w, int d, int f,
                                       uint8_t* __restrict__ packed) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  const int g = blockIdx.y;
  if (j >= f) return;
  const __half* col = w + (size_t)g * kGroup * f + j;
  float mx = -INFINITY, mn = INFINITY;
  for (int r = 0; r < kGroup; ++r) {
    const float v = __half2float(col[(size_t)r * f]);
    mx = fmaxf(mx, v);
    mn = fminf(mn, v);
  }
  __half s16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), 3.0f));
  if (__half2float(s16) == 0.0f) s16 = __float2half_rn(1.0f);
  const float sf = __half2float(s16);
  const float z32 = fminf(fmaxf(__fdiv_rn(-mn, sf), -65504.0f), 65504.0f);
  const __half z16 = __float2half_rn(z32);
  const int mt = j / kMTile, sb = g / 8, gi = g % 8;
  uint8_t* blk = packed + ((size_t)mt * n_superblocks(d) + sb) * kBlkBytes;
  __half2* sz = reinterpret_cast<__half2*>(blk + kBlkCodeBytes);
  sz[(j % kMTile) * 8 + gi] = __halves2half2(s16, z16);
}

// Entries of the (scale, zero) table for group slots past the end of d are zeroed.
__global__ void pack_clear_tail_kernel(int d, int f, uint8_t* __restrict__ packed) {
  const int mt = blockIdx.x;
  const int sb = n_superblocks(d) - 1;
  const int ng = (d - sb * kSuper) / kGroup;
  uint8_t* blk = packed + ((size_t)mt * n_superblocks(d) + sb) * kBlkBytes;
  uint32_t* sz = reinterpret_cast<uint32_t*>(blk + kBlkCodeBytes);
  const int t = threadIdx.x;  // 128 entries: 16 columns x 8 groups
  if (t < 128 && (t % 8) >= ng) sz[t] = 0u;
}

// One thread per packed code word: gathers its 16 codes.
__global__ void pack_codes_kernel(const __half* __restrict__ w, int d, int f,
                                  uint8_t* __restrict__ packed) {
  const int nsb = n_superblocks(d);
  const long long nwords = (long long)(f / kMTile) * nsb * 512;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= nwords) return;
  const int wi = (int)(idx & 3);
  const int lane = (int)((idx >> 2) & 31);
  const int u = (int)((idx >> 7) & 3);
  const long long blk_id = idx >> 9;
  const int sb = (int)(blk_id % nsb);
  const int mt = (int)(blk_id / nsb);
  const int gl = lane >> 2, c = lane & 3;
  const int j = mt * kMTile + gl + 8 * (wi & 1);
  uint8_t* blk = packed + (size_t)blk_id * kBlkBytes;
  const __half2* sz = reinterpret_cast<const __half2*>(blk + kBlkCodeBytes);
  uint32_t word = 0;
  for (int n = 0; n < 8; ++n) {
    const int g = sb * 8 + n;
    if (g * kGroup >= d) break;
    const __half2 p = sz[(j % kMTile) * 8 + n];
    const float sf = __low2float(p), zf = __high2float(p);
    for (int h = 0; h < 2; ++h) {
      const int k = sb * kSuper + n * kGroup + 16 * u + 2 * c + 8 * (wi >> 1) + h;
      const float v = __half2float(w[(size_t)k * f + j]);
      float q = rintf(__fadd_rn(__fdiv_rn(v, sf), zf));
      q = fminf(fmaxf(q, 0.0f), 3.0f);
      word |= (uint32_t)q << (2 * n + 16 * h);
    }
  }
  reinterpret_cast<uint32_t*>(blk)[(u * 32 + lane) * 4 + wi] = word;
}

// One thread per (k, j): canonical codes; one per (group, j): scale and zero.
__global__ void unpack_kernel(const uint8_t* __restrict__ packed, int d, int f,
                              uint8_t* __restrict__ q, __half* __restrict__ scale,
                              __half* __restrict__ zero) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)d * f) return;
  const int k = (int)(idx / f), j = (int)(idx % f);
  const int nsb = n_superblocks(d);
  const int sb = k / kSuper, n = (k % kSuper) / kGroup, kk = k % kGroup;
  const int u = kk / 16, r16 = kk % 16;
  const int h = r16 & 1, c = (r16 >> 1) & 3, rhi = r16 >> 3;
  const int mt = j / kMTile, jl = j % kMTile;
  const int gl = jl & 7, wi = rhi * 2 + (jl >> 3);
  const int lane = gl * 4 + c;
  const uint8_t* blk = packed + ((size_t)mt * nsb + sb) * kBlkBytes;
  const uint32_t word = reinterpret_cast<const uint32_t*>(blk)[(u * 32 + lane) * 4 + wi];
  if (q) q[idx] = (uint8_t)((word >> (2 * n + 16 * h)) & 3u);
  if (kk == 0) {
    const __half2 p = reinterpret_cast<const __half2*>(blk + kBlkCodeBytes)[jl * 8 + n];
    const size_t o = (size_t)(k / kGroup) * f + j;
    if (scale) scale[o] = __low2half(p);
    if (zero) zero[o] = __high2half(p);
  }
}

cudaError_t launch_pack(const __half* w, int d, int f, uint8_t* packed, cudaStream_t st) {
  dim3 g1((f + 127) / 128, d / kGroup);
  pack_scale_zero_kernel<<<g1, 128, 0, st>>>(w, d, f, packed);
  if (d % kSuper) pack_clear_tail_kernel<<<f / kMTile, 128, 0, st>>>(d, f, packed);
  const long long nwords = (long long)(f / kMTile) * n_superblocks(d) * 512;
  pack_codes_kernel<<<(unsigned)((nwords + 255) / 256), 256, 0, st>>>(w, d, f, packed);
  return cudaGetLastError();
}

cudaError_t launch_unpack(const uint8_t* packed, int d, int f, uint8_t* q, __half* scale,
                          __half* zero, cudaStream_t st) {
  const long long n = (long long)d * f;
  unpack_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(packed, d, f, q, scale, zero);
  return cudaGetLastError();
}

}  // namespace sesg
