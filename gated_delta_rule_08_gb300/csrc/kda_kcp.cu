// Context parallelism across devices: composing the affine maps of consecutive token ranges.
//
// Kimi K3: Open Frontier Intelligence (kimi-k3-paper.pages.dev), section 13.3.2 (KCP), and the
// open-day article (mlqm.cn), section 5.2: a long sequence is split into consecutive ranges, one
// per device.  Over a range the state pass is affine in its initial state,
//   S_out = P S_in + b   (P: the range's accumulated transition, b: its final state from S_in = 0),
// so after the devices exchange their fixed-size (P, b), each one folds the maps of the ranges
// before its own into its initial state:
//   S_in(0) = S0,  S_in(i + 1) = P_i S_in(i) + b_i.
// kda_state_compose evaluates that fold in fp32 on the device.  The per-range maps come from
// kda_chunk_fwd_segment_map (kda_scan_tc.cu, segment-map mode of the state pass).
//
//  compose_kernel (grid = heads x 32-column slices of the state, 256 threads): the slice of the
//  state lives in shared memory; per step P_i is staged in shared memory and every thread computes
//  dk / 8 entries of P_i S + b_i (lane = column, so P is read as warp-wide broadcasts and S
//  row-wise without bank conflicts).
#include <cuda_runtime.h>

#include "../../include/kda.h"
#include "kda_internal.h"

#define KDA_API extern "C" __attribute__((visibility("default")))

namespace kda {
namespace {

constexpr int kComposeThreads = 256;
constexpr int kSliceCols = 32;

template <int DK, int DV>
__global__ void __launch_bounds__(kComposeThreads) compose_kernel(const float* __restrict__ P,
                                                                  const float* __restrict__ b,
                                                                  const float* __restrict__ S0, float* S_out, int n,
                                                                  int H) {
  extern __shared__ float4 csm4[];
  float* sP = reinterpret_cast<float*>(csm4);  // [DK][DK]
  float* sS = sP + DK * DK;                    // [DK][kSliceCols]
  const int h = blockIdx.x, j0 = kSliceCols * blockIdx.y, tid = threadIdx.x;
  const int lane = tid & 31, rg = tid >> 5;  // column within the slice, row group
  constexpr int kRows = DK / 8;              // rows per thread: rg, rg + 8, ...
  const size_t soff = (size_t)h * DK * DV;
  for (int e = tid; e < DK * kSliceCols; e += kComposeThreads) {
    const int r = e / kSliceCols, c = e % kSliceCols;
    sS[e] = S0 != nullptr ? S0[soff + (size_t)r * DV + j0 + c] : 0.f;
  }
  for (int i = 0; i < n; ++i) {
    const float4* Pi = reinterpret_cast<const float4*>(P + ((size_t)i * H + h) * DK * DK);
    float4* sP4 = reinterpret_cast<float4*>(sP);
    for (int e = tid; e < DK * DK / 4; e += kComposeThreads) sP4[e] = Pi[e];
    const float* bi = b + ((size_t)i * H + h) * DK * DV;
    float acc[kRows];
#pragma unroll
    for (int j = 0; j < kRows; ++j) acc[j] = bi[(size_t)(rg + 8 * j) * DV + j0 + lane];
    __syncthreads();  // P_i staged; the previous step's state slice written
#pragma unroll 4
    for (int k = 0; k < DK; ++k) {
      const float s = sS[k * kSliceCols + lane];
#pragma unroll
      for (int j = 0; j < kRows; ++j) acc[j] = fmaf(sP[(rg + 8 * j) * DK + k], s, acc[j]);
    }
    __syncthreads();  // every read of sS and sP of this step is done
#pragma unroll
    for (int j = 0; j < kRows; ++j) sS[(rg + 8 * j) * kSliceCols + lane] = acc[j];
  }
  __syncthreads();
  for (int e = tid; e < DK * kSliceCols; e += kComposeThreads) {
    const int r = e / kSliceCols, c = e % kSliceCols;
    S_out[soff + (size_t)r * DV + j0 + c] = sS[e];
  }
}

template <int DK, int DV>
cudaError_t launch_compose(const float* P, const float* b, const float* S0, float* S_out, int n, int H,
                           cudaStream_t st) {
  static DeviceOnce once;
  constexpr size_t smem = (size_t)(DK * DK + DK * kSliceCols) * sizeof(float);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  const cudaError_t e = once.run(dev, [] {
    return cudaFuncSetAttribute(compose_kernel<DK, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  });
  if (e != cudaSuccess) return e;
  TraceScope ts("kda_state_compose", st);
  compose_kernel<DK, DV><<<dim3((unsigned)H, DV / kSliceCols), kComposeThreads, smem, st>>>(P, b, S0, S_out, n, H);
  return cudaGetLastError();
}

}  // namespace

cudaError_t state_compose_launch(const float* P, const float* b, const float* S0, float* S_out, int n, int H, int dk,
                                 int dv, cudaStream_t st) {
  if (dk == 128 && dv == 128) return launch_compose<128, 128>(P, b, S0, S_out, n, H, st);
  if (dk == 128 && dv == 64) return launch_compose<128, 64>(P, b, S0, S_out, n, H, st);
  if (dk == 64 && dv == 128) return launch_compose<64, 128>(P, b, S0, S_out, n, H, st);
  if (dk == 64 && dv == 64) return launch_compose<64, 64>(P, b, S0, S_out, n, H, st);
  return cudaErrorNotSupported;
}

}  // namespace kda
