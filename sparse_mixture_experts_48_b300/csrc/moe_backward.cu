// Backward pass of the layer (token choice): the kernels around the expert
// GEMMs.  Every sum runs in a fixed order, so gradients are bitwise
// reproducible.  Gradient of  L = sum_t <dy_t, y_t> + dL_aux * L_aux:
//
//   combine_bwd  per token: dO[slot(t,j)] = w_j dy_t, dw_j = <dy_t, O[slot(t,j)]>;
//                shared rows get dy_t.
//   router_bwd   per token: dl through the renormalised top-k weights
//                (softmax: w is the softmax of the selected logits, so
//                dl_i = w_i (dw_i - sum_j w_j dw_j); normalised sigmoid: through
//                the selected sigmoids) plus the L_aux term through P
//                (dp_te = dL_aux alpha E f_e / T).
//   dx           per token: sum of the grouped-row gradients of its kept
//                assignments (with expert choice: of the experts that chose
//                it) and shared experts, plus dl_t W_g^T (8 tokens per warp
//                share the W_g rows).
//   dWg          x^T dl and sum_t dl, in T-chunks, then the chunks in order.
//   colsum       bias gradients: column sums of dO / dA over a segment.
//   pad_zero     the padding rows of a grouped buffer (segments padded to
//                whole 128-row blocks for the weight-gradient GEMMs).
//
// Sources: "MoE混合专家模型：Transformer稀疏前馈网络原理与PyTorch实现" §4.3 (main and
// aux loss in one backward), §2.3 (Switch load-balance loss); "手撕一个极简
// MoE-FFN" §三 (renormalised top-k), §七 (f, P, L_aux); "MoE架构解析" §四
// 技术飞跃③ (normalised sigmoid gating).
#include <math.h>

#include "common.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

// ---- padding rows -------------------------------------------------------------
// Segment g's rows [out_row + real, out_row + rows) are zeroed (real = kept
// count for routed experts, T for shared ones).
__global__ void pad_zero_kernel(PadZeroArgs a) {
  const int g = blockIdx.x;
  const int64_t real = g < a.E ? a.counts[g] : a.T;
  const int64_t rows = a.seg.rows[g];
  const int64_t r0 = (int64_t)a.seg.out_row[g] + real;
  const int64_t npad = rows - real;
  if (npad <= 0) return;
  const int64_t chunks = a.row_bytes / 16;
  uint4* buf = (uint4*)a.buf;
  for (int64_t i = threadIdx.x; i < npad * chunks; i += blockDim.x)
    buf[(r0 + i / chunks) * chunks + i % chunks] = make_uint4(0u, 0u, 0u, 0u);
}

// ---- combine backward ----------------------------------------------------------
constexpr int kWarps = 4;

__global__ void __launch_bounds__(kWarps * 32) combine_bwd_kernel(CombineBwdArgs a) {
  const int lane = threadIdx.x % 32;
  const int64_t t = (int64_t)blockIdx.x * kWarps + threadIdx.x / 32;
  if (t >= a.T || *(volatile const uint32_t*)a.err != 0u) return;
  const int d = a.d, k = a.k;
  const uint16_t* dy = (const uint16_t*)a.dy + t * d;
  uint16_t* dO = (uint16_t*)a.dO;
  for (int j = 0; j < k; ++j) {
    const int slot = a.slot[t * k + j];
    if (slot < 0) {
      if (lane == 0) a.dw[t * k + j] = 0.f;
      continue;
    }
    const float w = a.topk_w[t * k + j];
    const float* o = a.o + (int64_t)slot * d;
    float dot = 0.f;
    for (int c = lane * 2; c < d; c += 64) {
      const uint32_t yy = *(const uint32_t*)(dy + c);
      const float y0 = bf16_bits_to_f32((uint16_t)(yy & 0xffffu)), y1 = bf16_bits_to_f32((uint16_t)(yy >> 16));
      const float2 ov = *(const float2*)(o + c);
      dot = fmaf(y0, ov.x, dot);
      dot = fmaf(y1, ov.y, dot);
      *(uint32_t*)(dO + (int64_t)slot * d + c) = pack_bf16x2(w * y0, w * y1);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
    if (lane == 0) a.dw[t * k + j] = dot;
  }
  for (int s = 0; s < a.S; ++s) {
    uint16_t* row = dO + (a.rows_routed + (int64_t)s * a.shared_stride + t) * d;
    for (int c = lane * 8; c < d; c += 256) *(uint4*)(row + c) = *(const uint4*)(dy + c);
  }
}

// ---- router backward -----------------------------------------------------------
__global__ void router_bwd_kernel(RouterBwdArgs a) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= a.T || *(volatile const uint32_t*)a.err != 0u) return;
  const int E = a.E, k = a.k;
  const float* l = a.logits + t * E;
  float* dl = a.dl + t * E;
  const bool soft = a.gating == MOE_GATE_SOFTMAX;
  // gate probabilities p over all E
  float mx = l[0];
  for (int e = 1; e < E; ++e) mx = fmaxf(mx, l[e]);
  float z = 0.f;
  for (int e = 0; e < E; ++e) z += soft ? expf(l[e] - mx) : 1.f / (1.f + expf(-l[e]));
  const float rz = 1.f / z;
  // aux term through P: dp_e = dL_aux alpha E (n_e / (T k)) / T
  const double cst = (double)a.dL_aux * a.alpha * (double)E / ((double)a.T * (double)a.T * (double)k);
  float pdp = 0.f;
  for (int e = 0; e < E; ++e) {
    const float pe = (soft ? expf(l[e] - mx) : 1.f / (1.f + expf(-l[e]))) * rz;
    pdp += pe * (float)(cst * (double)a.n_pre[e]);
  }
  for (int e = 0; e < E; ++e) {
    const float g = soft ? expf(l[e] - mx) : 1.f / (1.f + expf(-l[e]));
    const float pe = g * rz;
    const float dpe = (float)(cst * (double)a.n_pre[e]);
    // softmax: p (dp - <p, dp>); normalised sigmoid: (dp - <p, dp>) / sum s * s (1 - s)
    dl[e] = soft ? pe * (dpe - pdp) : (dpe - pdp) * rz * g * (1.f - g);
  }
  // selection term through the renormalised weights
  float wdw = 0.f, zsel = 0.f;
  for (int j = 0; j < k; ++j) {
    wdw += a.topk_w[t * k + j] * a.dw[t * k + j];
    if (!soft) zsel += 1.f / (1.f + expf(-l[a.topk_idx[t * k + j]]));
  }
  for (int j = 0; j < k; ++j) {
    const int e = a.topk_idx[t * k + j];
    const float w = a.topk_w[t * k + j], dwj = a.dw[t * k + j];
    if (soft) {
      dl[e] += w * (dwj - wdw);
    } else {
      const float s = 1.f / (1.f + expf(-l[e]));
      dl[e] += (dwj - wdw) / zsel * s * (1.f - s);
    }
  }
}

// ---- dx ---------------------------------------------------------------------------
// A warp handles kDxTok consecutive tokens, so every W_g row it loads (for the
// dl W_g^T term) serves all of them; a lane owns 4 consecutive columns.
constexpr int kMaxE = 256;

// Dynamic shared memory: s_dl [kWarps][kDxTok][E] gate-logit gradients, then
// with expert choice s_row [kWarps][kDxTok][E] the chosen rows of each token
// (ascending expert), listed once so that the column loop's loads of dxp do
// not wait on the bit mask and the row table.
template <int kDxTok>
__global__ void __launch_bounds__(kWarps * 32) dx_kernel(DxArgs a) {
  extern __shared__ float s_dyn[];
  __shared__ int s_slot[kWarps][kDxTok][8];
  __shared__ int s_nrow[kWarps][kDxTok];
  const int lane = threadIdx.x % 32, wl = threadIdx.x / 32;
  const int64_t t0 = ((int64_t)blockIdx.x * kWarps + wl) * kDxTok;
  if (t0 >= a.T || *(volatile const uint32_t*)a.err != 0u) return;
  const int d = a.d, k = a.k, E = a.E;
  float* s_dl = s_dyn + (int64_t)wl * kDxTok * E;                          // [kDxTok][E]
  int* s_row = (int*)(s_dyn + (int64_t)kWarps * kDxTok * E) + (int64_t)wl * kDxTok * E;   // [kDxTok][E]
  const int nt = a.T - t0 < kDxTok ? (int)(a.T - t0) : kDxTok;
  for (int i = lane; i < kDxTok * E; i += 32) {
    const int tt = i / E, e = i % E;
    s_dl[tt * E + e] = tt < nt ? a.dl[(t0 + tt) * E + e] : 0.f;
  }
  for (int i = lane; i < kDxTok * 8; i += 32) {
    const int tt = i / 8, j = i % 8;
    s_slot[wl][tt][j] = (tt < nt && j < k) ? a.slot[(t0 + tt) * k + j] : -1;
  }
  if (a.ec_bits) {
    const uint32_t lt = (1u << lane) - 1u;
    for (int tt = 0; tt < nt; ++tt) {
      const int64_t t = t0 + tt;
      int n = 0;
      for (int w = 0; w < a.EW; ++w) {
        const uint32_t m = a.ec_bits[t * a.EW + w];
        const int e = 32 * w + lane;
        if ((m >> lane) & 1u) s_row[tt * E + n + __popc(m & lt)] = a.ec_tok_row[t * E + e];
        n += __popc(m);
      }
      if (lane == 0) s_nrow[wl][tt] = n;
    }
  }
  __syncwarp();
  const uint16_t* Wg = (const uint16_t*)a.Wg;
  const bool wvec = (E % 8) == 0;   // rows of W_g in 16-byte pieces
  for (int c = 4 * lane; c < d; c += 128) {
    float r[kDxTok][4];
#pragma unroll
    for (int tt = 0; tt < kDxTok; ++tt)
#pragma unroll
      for (int q = 0; q < 4; ++q) r[tt][q] = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint16_t* wr = Wg + (int64_t)(c + q) * E;
      for (int e0 = 0; e0 < E; e0 += 8) {
        float wv[8];
        if (wvec) {
          const uint4 w = *reinterpret_cast<const uint4*>(wr + e0);
          const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            wv[2 * j] = __uint_as_float(ww[j] << 16);
            wv[2 * j + 1] = __uint_as_float(ww[j] & 0xffff0000u);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) wv[j] = e0 + j < E ? bf16_bits_to_f32(wr[e0 + j]) : 0.f;
        }
#pragma unroll
        for (int tt = 0; tt < kDxTok; ++tt)
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (e0 + j < E) r[tt][q] = fmaf(s_dl[tt * E + e0 + j], wv[j], r[tt][q]);
      }
    }
    for (int tt = 0; tt < nt; ++tt) {
      const int64_t t = t0 + tt;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int sl = s_slot[wl][tt][j];
        if (sl >= 0) {
          const float4 v = *reinterpret_cast<const float4*>(a.dxp + (int64_t)sl * d + c);
          acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
      }
      if (a.ec_bits) {
        // expert choice: the rows of the experts that chose t, ascending
        const int n = s_nrow[wl][tt];
        for (int j = 0; j < n; ++j) {
          const float4 v = *reinterpret_cast<const float4*>(a.dxp + (int64_t)s_row[tt * E + j] * d + c);
          acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
      }
      for (int s = 0; s < a.S; ++s) {
        const float4 v =
            *reinterpret_cast<const float4*>(a.dxp + (a.rows_routed + (int64_t)s * a.shared_stride + t) * d + c);
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
      }
      *reinterpret_cast<float4*>(a.dx + t * d + c) =
          make_float4(acc.x + r[tt][0], acc.y + r[tt][1], acc.z + r[tt][2], acc.w + r[tt][3]);
    }
  }
}

// ---- dW_g, db_g -------------------------------------------------------------------
constexpr int kDwgChunk = 256;   // tokens per chunk

// part[chunk][i][e] = sum_{t in chunk} x[t][i] dl[t][e];  bpart[chunk][e] = sum_{t in chunk} dl[t][e]
// kDwgEB experts per pass over the chunk.
template <int kDwgEB>
__global__ void dwg_partial_kernel(DwgArgs a) {
  __shared__ float s_dl[kDwgChunk][kDwgEB];
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t chunk = blockIdx.y;
  const int64_t t0 = chunk * kDwgChunk;
  const int64_t nt = a.T - t0 < kDwgChunk ? a.T - t0 : kDwgChunk;
  const uint16_t* x = (const uint16_t*)a.x;
  for (int e0 = 0; e0 < a.E; e0 += kDwgEB) {
    __syncthreads();
    for (int q = threadIdx.x; q < kDwgChunk * kDwgEB; q += blockDim.x) {
      const int tt = q / kDwgEB, ee = q % kDwgEB;
      s_dl[tt][ee] = (tt < nt && e0 + ee < a.E) ? a.dl[(t0 + tt) * a.E + e0 + ee] : 0.f;
    }
    __syncthreads();
    float acc[kDwgEB];
#pragma unroll
    for (int ee = 0; ee < kDwgEB; ++ee) acc[ee] = 0.f;
    if (i < a.d) {
      for (int tt = 0; tt < nt; ++tt) {
        const float xv = bf16_bits_to_f32(x[(t0 + tt) * a.d + i]);
#pragma unroll
        for (int ee = 0; ee < kDwgEB; ++ee) acc[ee] = fmaf(xv, s_dl[tt][ee], acc[ee]);
      }
#pragma unroll
      for (int ee = 0; ee < kDwgEB; ++ee)
        if (e0 + ee < a.E) a.part[(chunk * a.d + i) * a.E + e0 + ee] = acc[ee];
    }
    if (blockIdx.x == 0 && threadIdx.x < kDwgEB && e0 + threadIdx.x < a.E) {
      float s = 0.f;
      for (int tt = 0; tt < nt; ++tt) s += s_dl[tt][threadIdx.x];
      a.bpart[chunk * a.E + e0 + threadIdx.x] = s;
    }
  }
}

__global__ void dwg_final_kernel(DwgArgs a) {
  const int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t n = (int64_t)a.d * a.E;
  if (q < n) {
    float s = 0.f;
    for (int64_t ch = 0; ch < a.nchunk; ++ch) s += a.part[ch * n + q];
    a.dWg[q] = s;
  }
  if (a.dbg && q < a.E) {
    float s = 0.f;
    for (int64_t ch = 0; ch < a.nchunk; ++ch) s += a.bpart[ch * a.E + q];
    a.dbg[q] = s;
  }
}

// ---- bias gradients -----------------------------------------------------------------
__global__ void colsum_kernel(ColsumArgs a) {
  const int g = blockIdx.y;
  const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= a.N) return;
  const int64_t rows = a.seg.rows[g];
  const int64_t r0 = a.seg.out_row[g];
  const uint16_t* buf = (const uint16_t*)a.buf;
  float s = 0.f;
  for (int64_t r = 0; r < rows; ++r) s += bf16_bits_to_f32(buf[(r0 + r) * a.N + c]);
  a.out[(int64_t)a.seg.w[g] * a.N + c] = s;
}

}  // namespace

cudaError_t launch_pad_zero(const PadZeroArgs& a, cudaStream_t s) {
  if (a.G <= 0) return cudaSuccess;
  pad_zero_kernel<<<a.G, 256, 0, s>>>(a);
  return cudaGetLastError();
}
cudaError_t launch_combine_bwd(const CombineBwdArgs& a, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  combine_bwd_kernel<<<(unsigned)((a.T + kWarps - 1) / kWarps), kWarps * 32, 0, s>>>(a);
  return cudaGetLastError();
}
cudaError_t launch_router_bwd(const RouterBwdArgs& a, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  router_bwd_kernel<<<(unsigned)((a.T + 127) / 128), 128, 0, s>>>(a);
  return cudaGetLastError();
}
cudaError_t launch_dx(const DxArgs& a, cudaStream_t s) {
  if (a.T == 0) return cudaSuccess;
  if (a.E > kMaxE || a.k > 8) return cudaErrorInvalidValue;
  // Many experts make the dl W_g^T term heavy: 8 tokens per warp share the
  // W_g rows; with few experts one token per warp keeps more warps busy.
  const int lists = a.ec_bits ? 2 : 1;   // s_dl, and the chosen rows with expert choice
  if (a.E > 16) {
    const int64_t per_cta = (int64_t)kWarps * 8;
    const size_t smem = (size_t)lists * kWarps * 8 * a.E * 4;
    cudaError_t e = cudaFuncSetAttribute(dx_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dx_kernel<8><<<(unsigned)((a.T + per_cta - 1) / per_cta), kWarps * 32, smem, s>>>(a);
  } else {
    const size_t smem = (size_t)lists * kWarps * 1 * a.E * 4;
    dx_kernel<1><<<(unsigned)((a.T + kWarps - 1) / kWarps), kWarps * 32, smem, s>>>(a);
  }
  return cudaGetLastError();
}
int64_t dwg_chunks(int64_t T) { return (T + kDwgChunk - 1) / kDwgChunk; }
cudaError_t launch_dwg(const DwgArgs& a, cudaStream_t s) {
  if (a.T > 0) {
    dim3 grid((unsigned)((a.d + 127) / 128), (unsigned)a.nchunk);
    if (a.E <= 8)
      dwg_partial_kernel<8><<<grid, 128, 0, s>>>(a);
    else if (a.E <= 16)
      dwg_partial_kernel<16><<<grid, 128, 0, s>>>(a);
    else
      dwg_partial_kernel<32><<<grid, 128, 0, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const int64_t n = (int64_t)a.d * a.E;
  dwg_final_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(a);
  return cudaGetLastError();
}
cudaError_t launch_colsum(const ColsumArgs& a, cudaStream_t s) {
  if (a.G <= 0) return cudaSuccess;
  dim3 grid((unsigned)((a.N + 255) / 256), (unsigned)a.G);
  colsum_kernel<<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
