// Layout changes around the selective-scan kernels.  pad_rows / unpad_rows
// give rows of a ragged length the 16-byte aligned, vector-multiple layout of
// the vector path.  The others convert between the Mamba-2 token-major
// tensors and the channel-major rows of the scan, for the general Mamba-2 path
// (any head dim, up to 256 states, fp32 or bf16): a head of the Mamba-2
// recurrence of the Mamba-2 cuTile news page ("Технические детали
// оптимизации") is the selective scan of "Mamba CUDA 实现解析" eq (4)-(7)
// with the head's P channels as scan channels, A[d,n] = A_h for every state,
// the head's dt for every channel and the group's B/C rows.
//
//   to_rows:   in [nb][R][Cin] (token-major) -> out [G][nb][Cg][R] (rows of R
//              contiguous), Cout = Cin * rep channels split in G groups of Cg;
//              output channel c reads input column c / rep (rep > 1 broadcasts
//              a head's dt to its channels).
//   from_rows: the inverse for rep = 1: in [G][nb][Cg][R] -> out [nb][R][G*Cg].
//   group_rows: rows of W floats between [nb][G][Cg] and [G][nb][Cg] order
//              (the state of G > 1 groups).
// 32 x 32 tiles through shared memory, both sides coalesced.
#pragma once

#include <cstdint>

#include "ss_device.cuh"

namespace ss {

constexpr int kTile = 32;

template <typename T>
__global__ void __launch_bounds__(256) ss_to_rows(const T* __restrict__ in, T* __restrict__ out,
                                                   int64_t nb, int64_t R, int64_t Cin, int rep,
                                                   int64_t G) {
  __shared__ T tile[kTile][kTile + 1];
  const int64_t Cout = Cin * rep, Cg = Cout / G;
  const int64_t b = blockIdx.z;
  const int64_t r0 = (int64_t)blockIdx.y * kTile, c0 = (int64_t)blockIdx.x * kTile;
  const int tx = threadIdx.x % kTile, ty = threadIdx.x / kTile;  // 32 x 8 threads
  for (int i = ty; i < kTile; i += 8) {
    const int64_t r = r0 + i, c = c0 + tx;
    if (r < R && c < Cout) tile[i][tx] = in[(b * R + r) * Cin + c / rep];
  }
  __syncthreads();
  for (int i = ty; i < kTile; i += 8) {
    const int64_t c = c0 + i, r = r0 + tx;
    if (r < R && c < Cout) {
      const int64_t g = c / Cg, cc = c - g * Cg;
      out[((g * nb + b) * Cg + cc) * R + r] = tile[tx][i];
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(256) ss_from_rows(const T* __restrict__ in, T* __restrict__ out,
                                                     int64_t nb, int64_t R, int64_t C, int64_t G) {
  __shared__ T tile[kTile][kTile + 1];
  const int64_t Cg = C / G;
  const int64_t b = blockIdx.z;
  const int64_t r0 = (int64_t)blockIdx.y * kTile, c0 = (int64_t)blockIdx.x * kTile;
  const int tx = threadIdx.x % kTile, ty = threadIdx.x / kTile;
  for (int i = ty; i < kTile; i += 8) {
    const int64_t c = c0 + i, r = r0 + tx;
    if (r < R && c < C) {
      const int64_t g = c / Cg, cc = c - g * Cg;
      tile[i][tx] = in[((g * nb + b) * Cg + cc) * R + r];
    }
  }
  __syncthreads();
  for (int i = ty; i < kTile; i += 8) {
    const int64_t r = r0 + i, c = c0 + tx;
    if (r < R && c < C) out[(b * R + r) * C + c] = tile[tx][i];
  }
}

// to_group != 0: [nb][G][Cg][W] -> [G][nb][Cg][W]; else the inverse.
__global__ void ss_group_rows(const float* __restrict__ in, float* __restrict__ out, int64_t nb,
                              int64_t G, int64_t Cg, int64_t W, int to_group) {
  const int64_t total = nb * G * Cg * W;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t w = i % W, row = i / W;
    const int64_t cc = row % Cg, bg = row / Cg;  // bg: (b, g) or (g, b) of the source
    int64_t dst;
    if (to_group) {
      const int64_t g = bg % G, b = bg / G;
      dst = ((g * nb + b) * Cg + cc) * W + w;
    } else {
      const int64_t b = bg % nb, g = bg / nb;
      dst = ((b * G + g) * Cg + cc) * W + w;
    }
    out[dst] = in[i];
  }
}

// Per-head parameters repeated for the head's channels: A [H] -> [H*P][N],
// D, bias [H] -> [H*P] (null stays null).
__global__ void ss_expand_heads(const float* __restrict__ A, const float* __restrict__ D,
                                const float* __restrict__ bias, float* __restrict__ A_out,
                                float* __restrict__ D_out, float* __restrict__ bias_out,
                                int64_t H, int64_t P, int64_t N) {
  const int64_t total = H * P * N;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t c = i / N, h = c / P;
    A_out[i] = A[h];
    if (i % N == 0) {
      if (D) D_out[c] = D[h];
      if (bias) bias_out[c] = bias[h];
    }
  }
}

// Rows of a ragged length L copied into rows of Lp >= L steps (a multiple of
// the 16-byte vector) whose starts are 16-byte aligned, for the vector path:
// steps past L get `fill`, or, when `neg_of` is given, minus its entry for the
// row's channel (row % dim).  grid.y walks the rows, grid.x * block the
// vectors of a row; each thread writes whole 16-byte vectors.
template <typename T>
__global__ void __launch_bounds__(256) ss_pad_rows(const T* __restrict__ in, T* __restrict__ out,
                                                    int64_t rows, int64_t L, int64_t Lp,
                                                    float fill, const float* __restrict__ neg_of,
                                                    int64_t dim) {
  constexpr int V = Elem<T>::kVec;
  const int64_t nvec = Lp / V;
  for (int64_t row = blockIdx.y; row < rows; row += gridDim.y) {
    const T* src = in + row * L;
    T* dst = out + row * Lp;
    const T fv = Elem<T>::from_f32(neg_of ? -neg_of[row % dim] : fill);
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < nvec;
         v += (int64_t)gridDim.x * blockDim.x) {
      Vec16<T> w;
#pragma unroll
      for (int e = 0; e < V; ++e) {
        const int64_t t = v * V + e;
        w.e[e] = t < L ? src[t] : fv;
      }
      stg_vec(dst + v * V, w);
    }
  }
}

// ... and the first L steps of each padded row back into rows of L (whole
// 16-byte vectors read, elements written).
template <typename T>
__global__ void __launch_bounds__(256) ss_unpad_rows(const T* __restrict__ in, T* __restrict__ out,
                                                      int64_t rows, int64_t L, int64_t Lp) {
  constexpr int V = Elem<T>::kVec;
  const int64_t nvec = (L + V - 1) / V;
  for (int64_t row = blockIdx.y; row < rows; row += gridDim.y) {
    const T* src = in + row * Lp;
    T* dst = out + row * L;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < nvec;
         v += (int64_t)gridDim.x * blockDim.x) {
      const Vec16<T> w = ldg_vec(src + v * V);
#pragma unroll
      for (int e = 0; e < V; ++e) {
        const int64_t t = v * V + e;
        if (t < L) dst[t] = w.e[e];
      }
    }
  }
}

}  // namespace ss
