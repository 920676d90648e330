// e4m3 (8-bit) inputs, head dims 64, 128 and 256: the fused forward with
// Q K^T and P V on tcgen05.mma kind::f8f6f4, and the V transpose its P.V
// operand is read from when V is not read MN-major (kF8VMnMajor).
#include "launch.cuh"

namespace ea51 {

namespace {

// One CTA moves 128 keys x kTCols columns of one head: coalesced 16-byte
// loads of V rows into shared memory, then 16-byte stores of 16 consecutive
// keys of one column of V^T.  Keys in [N, n_pad) are written as zeros.
constexpr int kTKeys = 128;

template <int kTCols>
__global__ void __launch_bounds__(256) transpose_v8_kernel(const uint8_t* __restrict__ v,
                                                           uint8_t* __restrict__ vt, int N,
                                                           int n_pad, int nblk) {
  constexpr int kTPitch = kTCols + 4;  // bytes per staged row (breaks bank alignment)
  __shared__ __align__(16) uint8_t tile[kTKeys * kTPitch];
  const int key0 = static_cast<int>(blockIdx.x % static_cast<unsigned>(nblk)) * kTKeys;
  const size_t bh = blockIdx.x / static_cast<unsigned>(nblk);
  const uint8_t* src = v + (bh * N + key0) * kTCols;
  const int rows = min(kTKeys, N - key0);
  for (int i = threadIdx.x; i < kTKeys * (kTCols / 16); i += blockDim.x) {
    const int r = i / (kTCols / 16), c16 = i % (kTCols / 16);
    uint4 x = make_uint4(0u, 0u, 0u, 0u);
    if (r < rows) x = *reinterpret_cast<const uint4*>(src + static_cast<size_t>(r) * kTCols + c16 * 16);
    uint32_t* dst = reinterpret_cast<uint32_t*>(tile + r * kTPitch + c16 * 16);
    dst[0] = x.x;
    dst[1] = x.y;
    dst[2] = x.z;
    dst[3] = x.w;
  }
  __syncthreads();
  uint8_t* out = vt + bh * kTCols * static_cast<size_t>(n_pad);
  const int groups = (min(kTKeys, n_pad - key0) + 15) / 16;  // 16-key groups inside n_pad
  for (int i = threadIdx.x; i < kTCols * (kTKeys / 16); i += blockDim.x) {
    // a warp reads 32 consecutive columns of the same 16 staged rows
    const int c = i % kTCols, g = i / kTCols;
    if (g >= groups) continue;
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t x = 0;
#pragma unroll
      for (int b = 0; b < 4; ++b)
        x |= static_cast<uint32_t>(tile[(g * 16 + q * 4 + b) * kTPitch + c]) << (8 * b);
      w[q] = x;
    }
    *reinterpret_cast<uint4*>(out + static_cast<size_t>(c) * n_pad + key0 + g * 16) =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
}

template <int D>
cudaError_t launch_e4m3(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                        const CUtensorMap* to, const FwdParams& p, bool causal, cudaStream_t stream) {
  // split-KV partial outputs use their own instantiation, as for bf16
  if (p.kv_splits > 1)
    return causal ? launch_one<D, true, true, true>(tq, tk, tv, to, p, stream)
                  : launch_one<D, false, true, true>(tq, tk, tv, to, p, stream);
  return causal ? launch_one<D, true, false, true>(tq, tk, tv, to, p, stream)
                : launch_one<D, false, false, true>(tq, tk, tv, to, p, stream);
}

}  // namespace

cudaError_t launch_transpose_v8(const void* v, void* vt, long long BH, int N, int d, int n_pad,
                                cudaStream_t stream) {
  const long long nblk = (static_cast<long long>(N) + kTKeys - 1) / kTKeys;
  if ((d != 64 && d != 128 && d != 256) || N < 1 || n_pad % 16 != 0 || n_pad < N || BH < 1 ||
      BH * nblk > 0x7fffffffLL)
    return cudaErrorInvalidValue;
  const unsigned grid = static_cast<unsigned>(BH * nblk);
  if (d == 64)
    transpose_v8_kernel<64><<<grid, 256, 0, stream>>>(
        static_cast<const uint8_t*>(v), static_cast<uint8_t*>(vt), N, n_pad, static_cast<int>(nblk));
  else if (d == 128)
    transpose_v8_kernel<128><<<grid, 256, 0, stream>>>(
        static_cast<const uint8_t*>(v), static_cast<uint8_t*>(vt), N, n_pad, static_cast<int>(nblk));
  else
    transpose_v8_kernel<256><<<grid, 256, 0, stream>>>(
        static_cast<const uint8_t*>(v), static_cast<uint8_t*>(vt), N, n_pad, static_cast<int>(nblk));
  return cudaGetLastError();
}

FwdVariant fwd_variant_e4m3_d64() {
  using L = Layout<64, true>;
  return FwdVariant{L::BN, L::NQ * BM, &launch_e4m3<64>};
}

FwdVariant fwd_variant_e4m3_d128() {
  using L = Layout<128, true>;
  return FwdVariant{L::BN, L::NQ * BM, &launch_e4m3<128>};
}

FwdVariant fwd_variant_e4m3_d256() {
  using L = Layout<256, true>;
  return FwdVariant{L::BN, L::NQ * BM, &launch_e4m3<256>};
}

}  // namespace ea51
