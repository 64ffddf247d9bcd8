// Per-element GEMM epilogues shared by the SIMT and tensor-core kernels.
#pragma once

#include "gemm.h"

namespace ttt {

// Applies epilogue g.epi to accumulator `acc` of element (bz, m, n) and
// returns acc^2 for EPI_DW (the per-tile sum of squares feeding the
// per-sequence gradient norm), 0 otherwise.  S is the operand storage.
template <typename S>
__device__ __forceinline__ float epi_value(const GemmDesc& g, int bz, int m, int n, float acc) {
  using IO = OpIO<S>;
  switch (g.epi) {
    case EPI_STORE:
      IO::store(g.out, g.loO, bz * g.sO + (long long)m * g.ldo + n, acc);
      break;
    case EPI_STORE_F32:
      static_cast<float*>(g.out)[bz * g.sO + (long long)m * g.ldo + n] = acc;
      break;
    case EPI_GELU:
      if (g.out) IO::store(g.out, g.loO, bz * g.sO + (long long)m * g.ldo + n, acc);
      IO::store(g.out2, g.loO2, bz * g.sO2 + (long long)m * g.ldo2 + n, gelu_f(acc));
      break;
    case EPI_RESID: {
      const float r = static_cast<const float*>(g.aux)[bz * g.sX + (long long)m * g.ldx + n];
      const float v = r + acc;
      static_cast<float*>(g.out)[bz * g.sO + (long long)m * g.ldo + n] = v;
      if (g.out2) IO::store(g.out2, g.loO2, bz * g.sO2 + (long long)m * g.ldo2 + n, v);
      break;
    }
    case EPI_SWIGLU: {
      const float gt = static_cast<const float*>(g.aux)[bz * g.sX + (long long)m * g.ldx + n];
      IO::store(g.out, g.loO, bz * g.sO + (long long)m * g.ldo + n, silu_f(gt) * acc);
      break;
    }
    case EPI_DGELU: {
      const float z = IO::load(g.aux, g.loX, bz * g.sX + (long long)m * g.ldx + n);
      IO::store(g.out, g.loO, bz * g.sO + (long long)m * g.ldo + n, acc * gelu_grad_f(z));
      break;
    }
    case EPI_DW:
      OpIO<typename DwType<S>::T>::store(g.out, 0, bz * g.sO + (long long)m * g.ldo + n, acc);
      return acc * acc;
  }
  return 0.0f;
}

// Epilogue kind as a compile-time value; EK_ANY reads g.epi at run time.
constexpr int EK_ANY = -1;

// Pair version of epi_value for elements (m, n) and (m, n + 1), both inside
// the output (n even; every leading dim, batch stride and lo offset even).
// With EK fixed the compiler drops every other branch.
template <typename S, int EK>
__device__ __forceinline__ float epi_pair(const GemmDesc& g, int bz, int m, int n, float a0, float a1) {
  using P = PairIO<S>;
  const int ek = EK == EK_ANY ? (int)g.epi : EK;
  if (ek == EPI_STORE) {
    P::store(g.out, g.loO, bz * g.sO + (long long)m * g.ldo + n, a0, a1);
  } else if (ek == EPI_STORE_F32) {
    PairIO<float>::store(g.out, 0, bz * g.sO + (long long)m * g.ldo + n, a0, a1);
  } else if (ek == EPI_GELU) {
    if (g.out) P::store(g.out, g.loO, bz * g.sO + (long long)m * g.ldo + n, a0, a1);
    P::store(g.out2, g.loO2, bz * g.sO2 + (long long)m * g.ldo2 + n, gelu_f(a0), gelu_f(a1));
  } else if (ek == EPI_RESID) {
    const float2 r = PairIO<float>::load(g.aux, 0, bz * g.sX + (long long)m * g.ldx + n);
    const float v0 = r.x + a0, v1 = r.y + a1;
    PairIO<float>::store(g.out, 0, bz * g.sO + (long long)m * g.ldo + n, v0, v1);
    if (g.out2) P::store(g.out2, g.loO2, bz * g.sO2 + (long long)m * g.ldo2 + n, v0, v1);
  } else if (ek == EPI_SWIGLU) {
    const float2 gt = PairIO<float>::load(g.aux, 0, bz * g.sX + (long long)m * g.ldx + n);
    P::store(g.out, g.loO, bz * g.sO + (long long)m * g.ldo + n, silu_f(gt.x) * a0, silu_f(gt.y) * a1);
  } else if (ek == EPI_DGELU) {
    const float2 z = P::load(g.aux, g.loX, bz * g.sX + (long long)m * g.ldx + n);
    P::store(g.out, g.loO, bz * g.sO + (long long)m * g.ldo + n, a0 * gelu_grad_f(z.x), a1 * gelu_grad_f(z.y));
  } else if (ek == EPI_DW) {
    PairIO<typename DwType<S>::T>::store(g.out, 0, bz * g.sO + (long long)m * g.ldo + n, a0, a1);
    return a0 * a0 + a1 * a1;
  }
  return 0.0f;
}

}  // namespace ttt

namespace ttt {

// Eight consecutive elements i .. i+7 of a buffer at once (16-byte accesses;
// i, the base and, for Split, the lo offset are multiples of 8 elements).
template <typename S> struct OctIO;
template <> struct OctIO<float> {
  __device__ __forceinline__ static void load(const void* p, long long, long long i, float* v) {
    const float4* q = reinterpret_cast<const float4*>(static_cast<const float*>(p) + i);
    const float4 a = q[0], b = q[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
  __device__ __forceinline__ static void store(void* p, long long, long long i, const float* v) {
    float4* q = reinterpret_cast<float4*>(static_cast<float*>(p) + i);
    q[0] = make_float4(v[0], v[1], v[2], v[3]);
    q[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
};
template <> struct OctIO<bf16> {
  __device__ __forceinline__ static void load(const void* p, long long, long long i, float* v) {
    unpack_bf16x8(*reinterpret_cast<const uint4*>(static_cast<const bf16*>(p) + i), v);
  }
  __device__ __forceinline__ static void store(void* p, long long, long long i, const float* v) {
    *reinterpret_cast<uint4*>(static_cast<bf16*>(p) + i) = pack_bf16x8(v);
  }
};
template <> struct OctIO<Split> {
  __device__ __forceinline__ static void load(const void* p, long long lo, long long i, float* v) {
    const bf16* q = static_cast<const bf16*>(p);
    float h[8], l[8];
    unpack_bf16x8(*reinterpret_cast<const uint4*>(q + i), h);
    unpack_bf16x8(*reinterpret_cast<const uint4*>(q + lo + i), l);
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = h[j] + l[j];
  }
  __device__ __forceinline__ static void store(void* p, long long lo, long long i, const float* v) {
    bf16* q = static_cast<bf16*>(p);
    const uint4 hp = pack_bf16x8(v);
    float h[8], l[8];
    unpack_bf16x8(hp, h);
#pragma unroll
    for (int j = 0; j < 8; ++j) l[j] = v[j] - h[j];
    *reinterpret_cast<uint4*>(q + i) = hp;
    *reinterpret_cast<uint4*>(q + lo + i) = pack_bf16x8(l);
  }
};

// epi_value for the eight elements (m, n) .. (m, n+7) at once; requires
// GemmDesc::vec (every pointer, leading dim, batch stride and lo offset of the
// epilogue a multiple of 8 elements) and n + 8 <= N.  Returns the sum of acc^2
// for EPI_DW, 0 otherwise.
template <typename S, int EK>
__device__ __forceinline__ float epi_oct(const GemmDesc& g, int bz, int m, int n, const float* a) {
  using O = OctIO<S>;
  const int ek = EK == EK_ANY ? (int)g.epi : EK;
  const long long io = bz * g.sO + (long long)m * g.ldo + n;
  float t[8];
  if (ek == EPI_STORE) {
    O::store(g.out, g.loO, io, a);
  } else if (ek == EPI_STORE_F32) {
    OctIO<float>::store(g.out, 0, io, a);
  } else if (ek == EPI_GELU) {
    if (g.out) O::store(g.out, g.loO, io, a);
#pragma unroll
    for (int j = 0; j < 8; ++j) t[j] = gelu_f(a[j]);
    O::store(g.out2, g.loO2, bz * g.sO2 + (long long)m * g.ldo2 + n, t);
  } else if (ek == EPI_RESID) {
    OctIO<float>::load(g.aux, 0, bz * g.sX + (long long)m * g.ldx + n, t);
#pragma unroll
    for (int j = 0; j < 8; ++j) t[j] += a[j];
    OctIO<float>::store(g.out, 0, io, t);
    if (g.out2) O::store(g.out2, g.loO2, bz * g.sO2 + (long long)m * g.ldo2 + n, t);
  } else if (ek == EPI_SWIGLU) {
    OctIO<float>::load(g.aux, 0, bz * g.sX + (long long)m * g.ldx + n, t);
#pragma unroll
    for (int j = 0; j < 8; ++j) t[j] = silu_f(t[j]) * a[j];
    O::store(g.out, g.loO, io, t);
  } else if (ek == EPI_DGELU) {
    O::load(g.aux, g.loX, bz * g.sX + (long long)m * g.ldx + n, t);
#pragma unroll
    for (int j = 0; j < 8; ++j) t[j] = a[j] * gelu_grad_f(t[j]);
    O::store(g.out, g.loO, io, t);
  } else if (ek == EPI_DW) {
    OctIO<typename DwType<S>::T>::store(g.out, 0, io, a);
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) s += a[j] * a[j];
    return s;
  }
  return 0.0f;
}

}  // namespace ttt

namespace ttt {

// 32-byte (256-bit) global accesses: one whole sector per thread.  The address
// must be 32-byte aligned.
__device__ __forceinline__ void ld256(const void* p, uint32_t (&w)[8]) {
  asm volatile("ld.global.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
               : "l"(p));
}
__device__ __forceinline__ void st256(void* p, const uint32_t (&w)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]), "r"(w[1]),
               "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// Sixteen consecutive elements i .. i+15 at once with 32-byte accesses (i, the
// base and, for Split, the lo offset are multiples of 16 elements; bases
// 32-byte aligned).
template <typename S> struct HexIO;
template <> struct HexIO<float> {
  __device__ __forceinline__ static void load(const void* p, long long, long long i, float* v) {
    const float* q = static_cast<const float*>(p) + i;
    uint32_t w[8];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      ld256(q + 8 * h, w);
#pragma unroll
      for (int j = 0; j < 8; ++j) v[8 * h + j] = __uint_as_float(w[j]);
    }
  }
  __device__ __forceinline__ static void store(void* p, long long, long long i, const float* v) {
    float* q = static_cast<float*>(p) + i;
    uint32_t w[8];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int j = 0; j < 8; ++j) w[j] = __float_as_uint(v[8 * h + j]);
      st256(q + 8 * h, w);
    }
  }
};
__device__ __forceinline__ void pack_bf16x16(const float* v, uint32_t (&w)[8]) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
    w[j] = *reinterpret_cast<const uint32_t*>(&h);
  }
}
__device__ __forceinline__ void unpack_bf16x16(const uint32_t (&w)[8], float* v) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[j]));
    v[2 * j] = f.x;
    v[2 * j + 1] = f.y;
  }
}
template <> struct HexIO<bf16> {
  __device__ __forceinline__ static void load(const void* p, long long, long long i, float* v) {
    uint32_t w[8];
    ld256(static_cast<const bf16*>(p) + i, w);
    unpack_bf16x16(w, v);
  }
  __device__ __forceinline__ static void store(void* p, long long, long long i, const float* v) {
    uint32_t w[8];
    pack_bf16x16(v, w);
    st256(static_cast<bf16*>(p) + i, w);
  }
};
template <> struct HexIO<Split> {
  __device__ __forceinline__ static void load(const void* p, long long lo, long long i, float* v) {
    const bf16* q = static_cast<const bf16*>(p);
    uint32_t w[8];
    float l[16];
    ld256(q + i, w);
    unpack_bf16x16(w, v);
    ld256(q + lo + i, w);
    unpack_bf16x16(w, l);
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] += l[j];
  }
  __device__ __forceinline__ static void store(void* p, long long lo, long long i, const float* v) {
    bf16* q = static_cast<bf16*>(p);
    uint32_t w[8];
    float h[16], l[16];
    pack_bf16x16(v, w);
    unpack_bf16x16(w, h);
#pragma unroll
    for (int j = 0; j < 16; ++j) l[j] = v[j] - h[j];
    st256(q + i, w);
    pack_bf16x16(l, w);
    st256(q + lo + i, w);
  }
};

// epi_oct for sixteen elements (m, n) .. (m, n+15) with 32-byte accesses;
// requires GemmDesc::vec == 2 and n + 16 <= N.
template <typename S, int EK>
__device__ __forceinline__ float epi_hex(const GemmDesc& g, int bz, int m, int n, const float* a) {
  using O = HexIO<S>;
  const int ek = EK == EK_ANY ? (int)g.epi : EK;
  const long long io = bz * g.sO + (long long)m * g.ldo + n;
  float t[16];
  if (ek == EPI_STORE) {
    O::store(g.out, g.loO, io, a);
  } else if (ek == EPI_STORE_F32) {
    HexIO<float>::store(g.out, 0, io, a);
  } else if (ek == EPI_GELU) {
    if (g.out) O::store(g.out, g.loO, io, a);
#pragma unroll
    for (int j = 0; j < 16; ++j) t[j] = gelu_f(a[j]);
    O::store(g.out2, g.loO2, bz * g.sO2 + (long long)m * g.ldo2 + n, t);
  } else if (ek == EPI_RESID) {
    HexIO<float>::load(g.aux, 0, bz * g.sX + (long long)m * g.ldx + n, t);
#pragma unroll
    for (int j = 0; j < 16; ++j) t[j] += a[j];
    HexIO<float>::store(g.out, 0, io, t);
    if (g.out2) O::store(g.out2, g.loO2, bz * g.sO2 + (long long)m * g.ldo2 + n, t);
  } else if (ek == EPI_SWIGLU) {
    HexIO<float>::load(g.aux, 0, bz * g.sX + (long long)m * g.ldx + n, t);
#pragma unroll
    for (int j = 0; j < 16; ++j) t[j] = silu_f(t[j]) * a[j];
    O::store(g.out, g.loO, io, t);
  } else if (ek == EPI_DGELU) {
    O::load(g.aux, g.loX, bz * g.sX + (long long)m * g.ldx + n, t);
#pragma unroll
    for (int j = 0; j < 16; ++j) t[j] = a[j] * gelu_grad_f(t[j]);
    O::store(g.out, g.loO, io, t);
  } else if (ek == EPI_DW) {
    HexIO<typename DwType<S>::T>::store(g.out, 0, io, a);
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < 16; ++j) s += a[j] * a[j];
    return s;
  }
  return 0.0f;
}

}  // namespace ttt

namespace ttt {

// Epilogue kinds whose fp32 second input (aux) the tensor-core epilogue loads
// ahead of the accumulator (GELU' reads its z stash in place: prefetching it as
// well costs registers its arithmetic needs, measured slower).
template <int EK>
__host__ __device__ constexpr bool epi_reads_aux() {
  return EK == EPI_RESID || EK == EPI_SWIGLU;
}

// The aux values of elements (m, n) .. (m, n+15) as fp32 (32-byte loads; the
// same conditions as epi_hex).  Independent of the accumulator, so the
// tensor-core epilogue issues these loads before it waits for the MMAs.
template <typename S, int EK>
__device__ __forceinline__ void load_aux16(const GemmDesc& g, int bz, int m, int n, float* x) {
  const long long ix = bz * g.sX + (long long)m * g.ldx + n;
  if (EK == EPI_DGELU) HexIO<S>::load(g.aux, g.loX, ix, x);
  else HexIO<float>::load(g.aux, 0, ix, x);
}

// epi_hex with the aux values already loaded (x, fp32).
template <typename S, int EK>
__device__ __forceinline__ void epi_hex_x(const GemmDesc& g, int bz, int m, int n, const float* a, const float* x) {
  using O = HexIO<S>;
  const long long io = bz * g.sO + (long long)m * g.ldo + n;
  float t[16];
  if (EK == EPI_RESID) {
#pragma unroll
    for (int j = 0; j < 16; ++j) t[j] = x[j] + a[j];
    HexIO<float>::store(g.out, 0, io, t);
    if (g.out2) O::store(g.out2, g.loO2, bz * g.sO2 + (long long)m * g.ldo2 + n, t);
  } else if (EK == EPI_SWIGLU) {
#pragma unroll
    for (int j = 0; j < 16; ++j) t[j] = silu_f(x[j]) * a[j];
    O::store(g.out, g.loO, io, t);
  } else if (EK == EPI_DGELU) {
#pragma unroll
    for (int j = 0; j < 16; ++j) t[j] = a[j] * gelu_grad_f(x[j]);
    O::store(g.out, g.loO, io, t);
  }
}

}  // namespace ttt
