// quant.cu -- MX quantizer for sm_103a: real values -> FP8 / packed FP4 codes
// plus one E8M0 scale per block of K elements, the scales written straight
// into the atom layout the GEMM reads.
//
// Operation ("GEMM + RoPE + MXFP8 Projection (SM100)", section "Equations":
// MXFP8 quantize, an E8M0 per-block scale with E4M3 data; "GEMM + Amax
// (SM100)" for the scale atom layout and the E5M2 / packed E2M1 formats).  The
// pages do not spell out how a block's scale is chosen; the reading used takes
// the block's largest magnitude to the top binade of the element format:
//   amax = max |x| over the block, e = floor(log2 amax) - emax (E4M3 8,
//   E5M2 15, E2M1 2), e clamped to [-127, 127], scale byte e + 127,
//   code = round-to-nearest-even of x * 2^-e, saturated to the largest finite
//   value.  All-zero block: byte 127.  NaN or infinity in the block: byte 0xFF
//   and every code the format's NaN (E4M3 / E5M2 0x7F; E2M1 has none: 0).
//   Padding scale positions of the last atoms: byte 127.
//
// HBM-bound: one pass over X, coalesced 16-byte loads (4 fp32 or 8 bf16 per
// thread and chunk; eight fp32 or four bf16 chunks in flight per thread), the block maximum by
// shuffles among the 2..8 lanes sharing a block, packed round-to-nearest
// saturating conversions, coalesced code stores, one scale byte per block.

#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "bsgemm.h"
#include "bsquant.h"

namespace {

constexpr int kThreads = 256;
// chunks per thread per unit: 128 bytes of fp32 or 64 of bf16 in flight
__host__ __device__ constexpr int unroll_of(int in_bf16) { return in_bf16 ? 4 : 8; }
constexpr int kChunkBytes = 16;   // input bytes per thread per chunk

enum OutKind : int { kOutE4M3 = 0, kOutE5M2 = 1, kOutE2M1 = 2 };

// Division of a 32-bit n by an invariant d > 0 with one multiply-high and a
// shift (Granlund and Montgomery, "Division by invariant integers using
// multiplication", 1994): with s = ceil(log2 d) and m = floor(2^32 (2^s - d)
// / d) + 1, n / d = (mulhi(n, m) + n) >> s for every n < 2^32.
struct FastDiv {
  uint32_t d, m, s;
};

FastDiv make_fastdiv(uint32_t d) {
  FastDiv f;
  f.d = d;
  uint32_t s = 0;
  while ((uint64_t(1) << s) < d) ++s;
  f.s = s;
  f.m = static_cast<uint32_t>(((uint64_t(1) << 32) * ((uint64_t(1) << s) - d)) / d + 1);
  return f;
}

__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv& f) {
  return static_cast<uint32_t>((static_cast<uint64_t>(__umulhi(n, f.m)) + n) >> f.s);
}

struct QParams {
  const uint8_t* x;
  uint8_t* codes;
  uint8_t* sf;
  int64_t row_in_bytes;     // cols * input element size
  int64_t row_code_bytes;   // cols, or cols / 2 for E2M1
  uint32_t rows, cols, L;
  uint32_t chunks_per_row;  // cols / elements per chunk
  uint32_t num_units;       // L * rows * units_per_row (< 2^31)
  uint32_t nblk, t_r, t_k;  // blocks per row, atoms along rows and K
  FastDiv upr;              // units per row: ceil(chunks_per_row / (kThreads * unroll))
  FastDiv rows_div;         // rows
};

template <int OUT>
struct OutFmt;
template <>
struct OutFmt<kOutE4M3> { static constexpr int kEmax = 8; static constexpr uint32_t kNan = 0x7Fu; };
template <>
struct OutFmt<kOutE5M2> { static constexpr int kEmax = 15; static constexpr uint32_t kNan = 0x7Fu; };
template <>
struct OutFmt<kOutE2M1> { static constexpr int kEmax = 2; static constexpr uint32_t kNan = 0x0u; };

// Two values -> two codes, round to nearest even, saturating: `lo` in the
// low byte (FP8) or low nibble (FP4).
template <int OUT>
__device__ __forceinline__ uint32_t cvt2(float lo, float hi) {
  if (OUT == kOutE4M3) {
    uint16_t h;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(hi), "f"(lo));
    return h;
  } else if (OUT == kOutE5M2) {
    uint16_t h;
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(h) : "f"(hi), "f"(lo));
    return h;
  } else {
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return r;
  }
}

// Two fp32 products in one instruction (x.lo * y.lo, x.hi * y.hi).
__device__ __forceinline__ uint64_t mul2(uint64_t x, uint64_t y) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(x), "l"(y));
  return d;
}

// floor(log2 |v|) of a positive finite float given its magnitude bits.
__device__ __forceinline__ int floor_log2_bits(uint32_t a) {
  const int ef = static_cast<int>(a >> 23);
  if (ef > 0) return ef - 127;                  // normal: the unbiased exponent
  return (31 - __clz(static_cast<int>(a))) - 149;  // subnormal: a * 2^-149
}

// Byte offset of the scale of row `r`, block `kb`, batch `l` in the
// (L, t_r, t_k, 32, 4, 4) atom tensor (row r = 128 rt + 32 m1 + m0); the
// whole tensor is below 2^31 bytes.
__device__ __forceinline__ uint32_t sf_offset(uint32_t r, uint32_t kb, uint32_t l, uint32_t t_r,
                                              uint32_t t_k) {
  const uint32_t rt = r >> 7, rr = r & 127, kt = kb >> 2;
  return (((l * t_r + rt) * t_k + kt) << 9) + (rr & 31) * 16 + (rr >> 5) * 4 + (kb & 3);
}

template <int IN_BF16, int OUT, int SFV>
__global__ void __launch_bounds__(kThreads) bsq_quantize_kernel(const QParams p) {
  constexpr int E = IN_BF16 ? 8 : 4;   // elements per chunk
  constexpr int G = SFV / E;           // lanes per scale block (2..8)
  constexpr int kCodeBytes = OUT == kOutE2M1 ? E / 2 : E;
  constexpr int kUnroll = unroll_of(IN_BF16);
  using F = OutFmt<OUT>;
  const int tid = threadIdx.x;
  const int lane = tid & 31;

  for (uint32_t u = blockIdx.x; u < p.num_units; u += gridDim.x) {
    const uint32_t flat_row = fdiv(u, p.upr);
    const uint32_t seg = u - flat_row * p.upr.d;
    const uint32_t l = fdiv(flat_row, p.rows_div);
    const uint32_t r = flat_row - l * p.rows;
    const uint8_t* xrow = p.x + static_cast<int64_t>(flat_row) * p.row_in_bytes;
    uint8_t* crow = p.codes + static_cast<int64_t>(flat_row) * p.row_code_bytes;
    // all loads of the unit first, then the arithmetic
    uint4 raw[kUnroll];
    uint32_t ch[kUnroll];
#pragma unroll
    for (int i = 0; i < kUnroll; ++i) {
      ch[i] = (seg * kUnroll + i) * kThreads + tid;  // < 2^31: cols < 2^31
      raw[i] = ch[i] < p.chunks_per_row
                   ? __ldcs(reinterpret_cast<const uint4*>(xrow + static_cast<size_t>(ch[i]) * kChunkBytes))
                   : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int i = 0; i < kUnroll; ++i) {
      // a G-lane group holds one block, and is wholly in or out of the row
      const bool valid = ch[i] < p.chunks_per_row;
      float v[E];
      const uint32_t w[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
      if (IN_BF16) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          v[2 * j] = __uint_as_float(w[j] << 16);
          v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] = __uint_as_float(w[j]);
      }
      // block maximum of the magnitude bits (NaN and infinity order above
      // every finite value); bf16 pairs by a SIMD max of the 16-bit halves
      uint32_t amax = 0u;
      if (IN_BF16) {
        uint32_t m2 = 0u;
#pragma unroll
        for (int j = 0; j < 4; ++j) m2 = __vmaxu2(m2, w[j] & 0x7FFF7FFFu);
        amax = max(m2 & 0xFFFFu, m2 >> 16) << 16;
      } else {
#pragma unroll
        for (int j = 0; j < E; ++j) amax = max(amax, __float_as_uint(v[j]) & 0x7FFFFFFFu);
      }
#pragma unroll
      for (int off = 1; off < G; off <<= 1) amax = max(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
      if (!valid) continue;
      uint32_t byte = 127u;
      float inv = 1.0f;  // 2^-e
      const bool nonfinite = amax >= 0x7F800000u;
      if (nonfinite) {
        byte = 0xFFu;
      } else if (amax != 0u) {
        int e = floor_log2_bits(amax) - F::kEmax;
        e = min(max(e, -127), 127);
        byte = static_cast<uint32_t>(e + 127);
        // 2^-e as a float: normal for -e >= -126, the subnormal 2^-127 otherwise
        inv = -e >= -126 ? __uint_as_float(static_cast<uint32_t>(127 - e) << 23)
                         : __uint_as_float(0x00400000u);
      }
      uint32_t out[2] = {0u, 0u};
      if (nonfinite) {
        const uint32_t nan = F::kNan;
        if (OUT == kOutE2M1) {
          out[0] = 0u;
          out[1] = 0u;
        } else {
          out[0] = nan * 0x01010101u;
          out[1] = nan * 0x01010101u;
        }
      } else {
        // scaled pairs (exact: a power of two), then two codes per conversion
        const uint64_t inv2 = (static_cast<uint64_t>(__float_as_uint(inv)) << 32) | __float_as_uint(inv);
        float y[E];
#pragma unroll
        for (int j = 0; j < E / 2; ++j) {
          const uint64_t pr = (static_cast<uint64_t>(__float_as_uint(v[2 * j + 1])) << 32) |
                              __float_as_uint(v[2 * j]);
          const uint64_t sc = mul2(pr, inv2);
          y[2 * j] = __uint_as_float(static_cast<uint32_t>(sc));
          y[2 * j + 1] = __uint_as_float(static_cast<uint32_t>(sc >> 32));
        }
        if (OUT == kOutE2M1) {
          // E/2 bytes, element 2j in the low nibble of byte j
#pragma unroll
          for (int j = 0; j < E / 2; ++j)
            out[j / 4] |= cvt2<OUT>(y[2 * j], y[2 * j + 1]) << (8 * (j % 4));
        } else {
#pragma unroll
          for (int j = 0; j < E / 2; ++j)
            out[j / 2] |= cvt2<OUT>(y[2 * j], y[2 * j + 1]) << (16 * (j % 2));
        }
      }
      uint8_t* cdst = crow + static_cast<size_t>(ch[i]) * kCodeBytes;
      if (kCodeBytes == 8) *reinterpret_cast<uint2*>(cdst) = make_uint2(out[0], out[1]);
      else if (kCodeBytes == 4) *reinterpret_cast<uint32_t*>(cdst) = out[0];
      else *reinterpret_cast<uint16_t*>(cdst) = static_cast<uint16_t>(out[0]);
      if ((lane % G) == 0) p.sf[sf_offset(r, ch[i] / G, l, p.t_r, p.t_k)] = static_cast<uint8_t>(byte);
    }
  }

  // padding scale positions: rows past `rows` in the last row atoms, blocks
  // past `nblk` in the last K atoms (the loop above writes every other byte)
  const bool pad_rows = (p.rows & 127) != 0, pad_k = (p.nblk & 3) != 0;
  if (!pad_rows && !pad_k) return;
  const uint32_t atoms = p.L * (p.t_k + p.t_r);
  for (uint32_t a = blockIdx.x; a < atoms; a += gridDim.x) {
    const uint32_t l = a / (p.t_k + p.t_r);
    const uint32_t j = a - l * (p.t_k + p.t_r);
    uint32_t rt, kt;
    if (j < p.t_k) {
      if (!pad_rows) continue;
      rt = p.t_r - 1;
      kt = j;
    } else {
      if (!pad_k) continue;
      rt = j - p.t_k;
      kt = p.t_k - 1;
    }
    for (uint32_t b = tid; b < 512; b += kThreads) {
      const uint32_t m0 = b >> 4, m1 = (b >> 2) & 3, kin = b & 3;
      const uint32_t row = rt * 128 + m1 * 32 + m0, kb = kt * 4 + kin;
      if (row >= p.rows || kb >= p.nblk)
        p.sf[(((l * p.t_r + rt) * p.t_k + kt) << 9) + b] = 127u;
    }
  }
}

// ------------------------------------------------------------ columnwise
//
// The S-direction of the same rule ("GEMM + RoPE + MXFP8 Projection (SM100)",
// sections "Overview" and "Equations": blocks along the tokens, the
// non-contiguous dimension): X (L, rows, cols), cols contiguous, one E8M0
// scale per 32 consecutive rows of a column.  The codes keep X's layout --
// the GEMM's MN-major operand with rows as K -- and the scale of (column c,
// block b) goes where the GEMM reads row mn = c, K-block kb = b of the atom
// tensor (L, ceil(cols/128), ceil(rows/128), 32, 4, 4).  FP8 codes only.
//
// A unit is one 128-row atom of K by 8 warps x kColsPerWarp columns.  Within
// a 32-row block, lane t of a warp holds rows t/8 + 4i (i < 8) of the 16-byte
// column chunk t%8, so each load instruction reads four rows of 128
// contiguous bytes; the four lanes sharing a chunk combine their column
// maxima by two shuffles.  After the unit's four blocks, lanes 0..7 write
// each column's four scale bytes (K-blocks 0..3 of the atom) as one 32-bit
// word; columns past `cols` and blocks past rows/32 keep byte 127.

struct QCParams {
  const uint8_t* x;
  uint8_t* codes;
  uint8_t* sf;
  uint32_t rows, cols, L;
  uint32_t nblk, t_c, t_k;  // blocks per column (rows / 32); atoms along cols and rows
  uint32_t num_units;       // L * t_k * col_units
  FastDiv cu_div;           // column units per atom row: ceil(cols / unit columns)
  FastDiv tk_div;           // t_k
};

template <int IN_BF16>
struct ColTile {
  static constexpr int kE = IN_BF16 ? 8 : 4;           // columns per 16-byte chunk
  static constexpr int kColsPerWarp = 8 * kE;           // 8 chunk lanes x kE
  static constexpr int kUnitCols = 8 * kColsPerWarp;    // 8 warps
};

// Loads in flight (bf16 input): each thread copies its eight 16-byte row
// pieces of a block into its own slots of a shared ring (cp.async, zero-filled
// past `cols`) and keeps kColStages - 1 blocks in flight ahead of the one it
// converts, so the bytes in flight no longer depend on registers: the bf16
// conversion needs ~112 registers, two CTAs per SM, and loading through
// registers left half the fp32 kernel's bytes in flight (67 % of the copy
// bandwidth, against 77 % this way).  A thread reads back only what it copied
// itself, so no barrier is needed.  fp32 input (64 registers, four CTAs per
// SM) already keeps enough in flight through registers and loads directly.
constexpr int kColStages = 3;
constexpr int kColStageBytes = 8 * kThreads * 16;  // one block: 8 row pieces per thread
constexpr int kColSmemBytes = kColStages * kColStageBytes;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// One block of 32 rows of this thread's columns (its eight row pieces in
// raw, zero past `cols`): the column maxima over the block, the scale bytes
// (into byte b of sfw), the codes.
template <int IN_BF16, int OUT>
__device__ __forceinline__ void colwise_block(const QCParams& p, const uint4 (&raw)[8], uint32_t l,
                                              uint32_t row0, uint32_t b, uint32_t c0, bool col_ok,
                                              uint32_t (&sfw)[ColTile<IN_BF16>::kE]) {
  constexpr int E = ColTile<IN_BF16>::kE;
  using F = OutFmt<OUT>;
  // per column: max of the magnitude bits over this lane's 8 rows, then
  // over the 4 row groups (NaN and infinity order above every finite value).
  // bf16: a SIMD max of the packed 16-bit magnitudes (they order like the
  // fp32 bits they widen to), two columns per word.
  uint32_t amax[E];
  if constexpr (IN_BF16) {
    uint32_t m2[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t w[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) m2[k] = __vmaxu2(m2[k], w[k] & 0x7FFF7FFFu);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      m2[k] = __vmaxu2(m2[k], __shfl_xor_sync(0xFFFFFFFFu, m2[k], 8));
      m2[k] = __vmaxu2(m2[k], __shfl_xor_sync(0xFFFFFFFFu, m2[k], 16));
    }
#pragma unroll
    for (int j = 0; j < E; ++j) amax[j] = (j & 1) ? (m2[j / 2] & 0xFFFF0000u) : (m2[j / 2] << 16);
  } else {
#pragma unroll
    for (int j = 0; j < E; ++j) amax[j] = 0u;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t w[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
      for (int j = 0; j < E; ++j) amax[j] = max(amax[j], w[j] & 0x7FFFFFFFu);
    }
#pragma unroll
    for (int j = 0; j < E; ++j) {
      amax[j] = max(amax[j], __shfl_xor_sync(0xFFFFFFFFu, amax[j], 8));
      amax[j] = max(amax[j], __shfl_xor_sync(0xFFFFFFFFu, amax[j], 16));
    }
  }
  if (!col_ok) return;  // a chunk past `cols`: it only took part in the shuffles
  float inv[E];
  bool nonfinite[E];
#pragma unroll
  for (int j = 0; j < E; ++j) {
    uint32_t byte = 127u;
    inv[j] = 1.0f;
    nonfinite[j] = amax[j] >= 0x7F800000u;
    if (nonfinite[j]) {
      byte = 0xFFu;
    } else if (amax[j] != 0u) {
      int e = floor_log2_bits(amax[j]) - F::kEmax;
      e = min(max(e, -127), 127);
      byte = static_cast<uint32_t>(e + 127);
      inv[j] = -e >= -126 ? __uint_as_float(static_cast<uint32_t>(127 - e) << 23)
                          : __uint_as_float(0x00400000u);
    }
    sfw[j] = (sfw[j] & ~(0xFFu << (8 * b))) | (byte << (8 * b));
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t w[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
    float v[E];
#pragma unroll
    for (int j = 0; j < E; ++j)
      v[j] = __uint_as_float(IN_BF16 ? ((j & 1) ? (w[j / 2] & 0xFFFF0000u) : (w[j / 2] << 16))
                                     : w[j]);
    uint32_t out[E / 4];
#pragma unroll
    for (int k = 0; k < E / 4; ++k) out[k] = 0u;
#pragma unroll
    for (int j = 0; j < E; j += 2) {
      // exact products (powers of two, a pair per multiply), then two codes
      // per conversion
      const uint64_t pr = (static_cast<uint64_t>(__float_as_uint(v[j + 1])) << 32) | __float_as_uint(v[j]);
      const uint64_t iv = (static_cast<uint64_t>(__float_as_uint(inv[j + 1])) << 32) | __float_as_uint(inv[j]);
      const uint64_t sc = mul2(pr, iv);
      uint32_t c2 = cvt2<OUT>(__uint_as_float(static_cast<uint32_t>(sc)),
                              __uint_as_float(static_cast<uint32_t>(sc >> 32)));
      if (nonfinite[j]) c2 = (c2 & 0xFF00u) | F::kNan;
      if (nonfinite[j + 1]) c2 = (c2 & 0x00FFu) | (F::kNan << 8);
      out[j / 4] |= c2 << (16 * ((j / 2) % 2));
    }
    uint8_t* dst = p.codes + (static_cast<size_t>(l) * p.rows + row0 + 4 * i) * p.cols + c0;
    if (E == 8) *reinterpret_cast<uint2*>(dst) = make_uint2(out[0], out[E / 4 - 1]);
    else *reinterpret_cast<uint32_t*>(dst) = out[0];
  }
}

// A unit's scale words: lanes of row group 0, one word per column of a real
// atom (columns past `cols` in the last atom: padding 127).
template <int IN_BF16>
__device__ __forceinline__ void colwise_scale_words(const QCParams& p, uint32_t l, uint32_t kt,
                                                    uint32_t c0, int rg,
                                                    const uint32_t (&sfw)[ColTile<IN_BF16>::kE]) {
  if (rg != 0) return;
#pragma unroll
  for (int j = 0; j < ColTile<IN_BF16>::kE; ++j) {
    const uint32_t c = c0 + j;
    const uint32_t atom = c >> 7;
    if (atom < p.t_c) {
      const uint32_t off = (((l * p.t_c + atom) * p.t_k + kt) << 9) + (c & 31) * 16 + ((c & 127) >> 5) * 4;
      *reinterpret_cast<uint32_t*>(p.sf + off) = sfw[j];
    }
  }
}

// fp32 input: loads through registers, eight 16-byte row pieces per block in
// flight per thread, four CTAs per SM.
template <int OUT>
__device__ __forceinline__ void colwise_direct(const QCParams& p) {
  using T = ColTile<0>;
  constexpr int E = T::kE;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int chunk = lane & 7, rg = lane >> 3;  // column chunk of the warp, row group
  for (uint32_t u = blockIdx.x; u < p.num_units; u += gridDim.x) {
    const uint32_t lk = fdiv(u, p.cu_div);  // l * t_k + kt
    const uint32_t cu = u - lk * p.cu_div.d;
    const uint32_t l = fdiv(lk, p.tk_div);
    const uint32_t kt = lk - l * p.t_k;
    const uint32_t c0 = cu * T::kUnitCols + warp * T::kColsPerWarp + chunk * E;
    const bool col_ok = c0 < p.cols;  // cols % 16 == 0: a chunk is wholly in or out
    const uint32_t nb = min(4u, p.nblk - kt * 4);
    uint32_t sfw[E];
#pragma unroll
    for (int j = 0; j < E; ++j) sfw[j] = 0x7F7F7F7Fu;
    for (uint32_t b = 0; b < nb; ++b) {
      const uint32_t row0 = kt * 128 + b * 32 + rg;
      uint4 raw[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const size_t e = (static_cast<size_t>(l) * p.rows + row0 + 4 * i) * p.cols + c0;
        raw[i] = col_ok ? __ldcs(reinterpret_cast<const uint4*>(p.x + e * 4))
                        : make_uint4(0u, 0u, 0u, 0u);
      }
      colwise_block<0, OUT>(p, raw, l, row0, b, c0, col_ok, sfw);
    }
    colwise_scale_words<0>(p, l, kt, c0, rg, sfw);
  }
}

// bf16 input: the load ring (above).
template <int OUT>
__device__ __forceinline__ void colwise_ring(const QCParams& p) {
  using T = ColTile<1>;
  constexpr int E = T::kE;
  extern __shared__ __align__(16) uint8_t qc_ring[];
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int chunk = lane & 7, rg = lane >> 3;  // column chunk of the warp, row group
  // this thread's piece i of ring slot s (consecutive threads, consecutive 16 bytes)
  const uint32_t ring0 = static_cast<uint32_t>(__cvta_generic_to_shared(qc_ring)) + tid * 16u;
  auto slot_addr = [&](int s, int i) { return ring0 + static_cast<uint32_t>((s * 8 + i) * kThreads * 16); };
  // a position in this CTA's walk over (unit, block of 32 rows)
  struct Cursor {
    uint32_t u, b, nb, l, kt, c0;
    bool col_ok, valid;
  };
  auto set_unit = [&](Cursor& c, uint32_t u) {
    c.u = u;
    c.b = 0;
    c.valid = u < p.num_units;
    if (!c.valid) return;
    const uint32_t lk = fdiv(u, p.cu_div);  // l * t_k + kt
    const uint32_t cu = u - lk * p.cu_div.d;
    c.l = fdiv(lk, p.tk_div);
    c.kt = lk - c.l * p.t_k;
    c.c0 = cu * T::kUnitCols + warp * T::kColsPerWarp + chunk * E;
    c.col_ok = c.c0 < p.cols;  // cols % 16 == 0: a chunk is wholly in or out
    c.nb = min(4u, p.nblk - c.kt * 4);
  };
  auto advance = [&](Cursor& c) {
    if (++c.b == c.nb) set_unit(c, c.u + gridDim.x);
  };
  // the copies of the cursor's block into ring slot s (one commit group)
  auto issue = [&](const Cursor& c, int s) {
    if (c.valid) {
      const uint32_t row0 = c.kt * 128 + c.b * 32 + rg;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const size_t e = (static_cast<size_t>(c.l) * p.rows + row0 + 4 * i) * p.cols + c.c0;
        cp_async16(slot_addr(s, i), c.col_ok ? static_cast<const void*>(p.x + e * 2) : p.x,
                   c.col_ok ? 16u : 0u);
      }
    }
    cp_async_commit();
  };
  Cursor ld, cur;
  set_unit(ld, blockIdx.x);
  cur = ld;
#pragma unroll
  for (int s = 0; s < kColStages - 1; ++s) {
    issue(ld, s);
    if (ld.valid) advance(ld);
  }
  int slot = 0;
  uint32_t sfw[E];  // per column: the scale bytes of K-blocks 0..3 of this atom
#pragma unroll
  for (int j = 0; j < E; ++j) sfw[j] = 0x7F7F7F7Fu;
  while (cur.valid) {
    issue(ld, slot == 0 ? kColStages - 1 : slot - 1);
    if (ld.valid) advance(ld);
    cp_async_wait<kColStages - 1>();  // this block's copies have landed
    uint4 raw[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint4 v;
      asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                   : "r"(slot_addr(slot, i)));
      raw[i] = v;
    }
    colwise_block<1, OUT>(p, raw, cur.l, cur.kt * 128 + cur.b * 32 + rg, cur.b, cur.c0, cur.col_ok, sfw);
    if (cur.b + 1 == cur.nb) {  // the unit's last block
      colwise_scale_words<1>(p, cur.l, cur.kt, cur.c0, rg, sfw);
#pragma unroll
      for (int j = 0; j < E; ++j) sfw[j] = 0x7F7F7F7Fu;
    }
    advance(cur);
    slot = slot == kColStages - 1 ? 0 : slot + 1;
  }
  cp_async_wait<0>();  // no copy of this thread outlives it
}

template <int IN_BF16, int OUT>
__global__ void __launch_bounds__(kThreads) bsq_quantize_colwise_kernel(const QCParams p) {
  if constexpr (IN_BF16) colwise_ring<OUT>(p);
  else colwise_direct<OUT>(p);
}

template <int IN_BF16, int OUT, int SFV>
const void* kernel_of() {
  return reinterpret_cast<const void*>(&bsq_quantize_kernel<IN_BF16, OUT, SFV>);
}

// variant index for the per-device occupancy cache: [in_bf16][E4M3, E5M2, E2M1/16, E2M1/32]
int variant_of(int in_bf16, int out, int sfv) {
  return in_bf16 * 4 + (out == kOutE2M1 ? (sfv == 16 ? 2 : 3) : out);
}

template <int IN_BF16, int OUT>
const void* colwise_kernel_of() {
  return reinterpret_cast<const void*>(&bsq_quantize_colwise_kernel<IN_BF16, OUT>);
}

const void* pick_colwise_kernel(int in_bf16, int out) {
  if (out == kOutE4M3) return in_bf16 ? colwise_kernel_of<1, kOutE4M3>() : colwise_kernel_of<0, kOutE4M3>();
  return in_bf16 ? colwise_kernel_of<1, kOutE5M2>() : colwise_kernel_of<0, kOutE5M2>();
}

const void* pick_kernel(int in_bf16, int out, int sfv) {
  if (out == kOutE4M3) return in_bf16 ? kernel_of<1, kOutE4M3, 32>() : kernel_of<0, kOutE4M3, 32>();
  if (out == kOutE5M2) return in_bf16 ? kernel_of<1, kOutE5M2, 32>() : kernel_of<0, kOutE5M2, 32>();
  if (sfv == 16) return in_bf16 ? kernel_of<1, kOutE2M1, 16>() : kernel_of<0, kOutE2M1, 16>();
  return in_bf16 ? kernel_of<1, kOutE2M1, 32>() : kernel_of<0, kOutE2M1, 32>();
}

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
int g_dev_sms[kMaxDevices] = {};   // 0: not queried yet; -1: not an sm_103 device
// resident CTAs per SM of each variant (0: not queried): rowwise [0, 8) as
// variant_of, columnwise 8 + in_bf16 * 2 + out (E4M3 0, E5M2 1)
int g_dev_occ[kMaxDevices][12] = {};

// One launch of the columnwise kernel (the request already checked).
bsg_status launch_colwise(const bsg_quant_problem* q, const void* X, void* codes, void* sf,
                          void* stream, int dev, int sms) {
  QCParams p;
  std::memset(&p, 0, sizeof(p));
  const int in_bf16 = q->in_dtype == BSG_BF16 ? 1 : 0;
  const int out = q->out_dtype == BSG_E4M3 ? kOutE4M3 : kOutE5M2;
  p.x = static_cast<const uint8_t*>(X);
  p.codes = static_cast<uint8_t*>(codes);
  p.sf = static_cast<uint8_t*>(sf);
  p.rows = static_cast<uint32_t>(q->rows);
  p.cols = static_cast<uint32_t>(q->cols);
  p.L = static_cast<uint32_t>(q->L);
  p.nblk = p.rows / 32;
  p.t_c = static_cast<uint32_t>(cdiv(q->cols, 128));
  p.t_k = static_cast<uint32_t>(cdiv(p.nblk, 4));
  const int64_t unit_cols = in_bf16 ? ColTile<1>::kUnitCols : ColTile<0>::kUnitCols;
  const int64_t col_units = cdiv(q->cols, unit_cols);
  const int64_t units = q->L * static_cast<int64_t>(p.t_k) * col_units;
  if (units > (int64_t(1) << 31) - 1) return BSG_ERR_INVALID_ARG;
  p.num_units = static_cast<uint32_t>(units);
  p.cu_div = make_fastdiv(static_cast<uint32_t>(col_units));
  p.tk_div = make_fastdiv(p.t_k);
  const void* fn = pick_colwise_kernel(in_bf16, out);
  const int ring_bytes = in_bf16 ? kColSmemBytes : 0;  // the bf16 kernel's load ring
  int occ;
  {
    std::lock_guard<std::mutex> lock(g_dev_mu);
    int& slot = g_dev_occ[dev][8 + in_bf16 * 2 + out];
    if (slot == 0) {
      int n = 0;
      if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, ring_bytes) !=
              cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kThreads, ring_bytes) != cudaSuccess) {
        cudaGetLastError();
        return BSG_ERR_CUDA;
      }
      slot = n < 1 ? 1 : (n > 8 ? 8 : n);
    }
    occ = slot;
  }
  int64_t grid = static_cast<int64_t>(sms) * occ;
  if (grid > p.num_units) grid = p.num_units;
  void* args[1] = {&p};
  if (cudaLaunchKernel(fn, dim3(static_cast<unsigned>(grid)), dim3(kThreads), args, ring_bytes,
                       static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return BSG_ERR_CUDA;
  }
  return BSG_OK;
}

}  // namespace

extern "C" {

bsg_status bsg_quant_check(const bsg_quant_problem* q) {
  if (!q) return BSG_ERR_INVALID_ARG;
  const int64_t lim = (int64_t(1) << 31) - 1;
  if (q->rows < 1 || q->cols < 1 || q->L < 1) return BSG_ERR_INVALID_ARG;
  if (q->rows > lim || q->cols > lim || q->L > lim || q->rows * q->L > lim)
    return BSG_ERR_INVALID_ARG;
  if (q->direction != BSG_QUANT_ROWWISE && q->direction != BSG_QUANT_COLWISE)
    return BSG_ERR_INVALID_ARG;
  if (q->direction == BSG_QUANT_COLWISE) {
    // blocks of 32 rows down each column; FP8 codes (the GEMM's MN-major
    // operands are FP8 only); code rows of `cols` bytes 16-byte aligned
    if (q->in_dtype != BSG_F32 && q->in_dtype != BSG_BF16) return BSG_ERR_INVALID_ARG;
    if (q->out_dtype != BSG_E4M3 && q->out_dtype != BSG_E5M2 && q->out_dtype != BSG_E2M1)
      return BSG_ERR_INVALID_ARG;
    if (q->sf_vec_size != 16 && q->sf_vec_size != 32) return BSG_ERR_INVALID_ARG;
    if (q->out_dtype == BSG_E2M1 || q->sf_vec_size != 32) return BSG_ERR_UNSUPPORTED;
    if (q->rows % 32 != 0) return BSG_ERR_UNSUPPORTED;  // whole blocks only
    if (q->cols % 16 != 0) return BSG_ERR_ALIGNMENT;
    const int64_t sf_bytes = q->L * ((q->cols + 127) / 128) * ((q->rows / 32 + 3) / 4) * 512;
    if (sf_bytes > lim || q->L * q->rows * q->cols / 16 > lim) return BSG_ERR_INVALID_ARG;
    return BSG_OK;
  }
  // the scale atom tensor is indexed with 32-bit offsets
  if (q->sf_vec_size == 16 || q->sf_vec_size == 32) {
    const int64_t sf_bytes =
        q->L * ((q->rows + 127) / 128) * ((q->cols / q->sf_vec_size + 3) / 4) * 512;
    if (sf_bytes > lim) return BSG_ERR_INVALID_ARG;
  }
  if (q->in_dtype != BSG_F32 && q->in_dtype != BSG_BF16) return BSG_ERR_INVALID_ARG;
  if (q->out_dtype != BSG_E4M3 && q->out_dtype != BSG_E5M2 && q->out_dtype != BSG_E2M1)
    return BSG_ERR_INVALID_ARG;
  if (q->sf_vec_size != 16 && q->sf_vec_size != 32) return BSG_ERR_INVALID_ARG;
  if (q->out_dtype != BSG_E2M1 && q->sf_vec_size != 32) return BSG_ERR_UNSUPPORTED;
  if (q->cols % q->sf_vec_size != 0) return BSG_ERR_UNSUPPORTED;  // whole blocks only
  return BSG_OK;
}

bsg_status bsg_quant_sizes(const bsg_quant_problem* q, size_t* code_bytes, size_t* sf_bytes) {
  const bsg_status st = bsg_quant_check(q);
  if (st != BSG_OK) return st;
  if (!code_bytes || !sf_bytes) return BSG_ERR_INVALID_ARG;
  if (q->direction == BSG_QUANT_COLWISE) {
    *code_bytes = static_cast<size_t>(q->L * q->rows * q->cols);
    *sf_bytes = static_cast<size_t>(q->L * cdiv(q->cols, 128) * cdiv(q->rows / 32, 4) * 512);
    return BSG_OK;
  }
  const int64_t per_row = q->out_dtype == BSG_E2M1 ? q->cols / 2 : q->cols;
  *code_bytes = static_cast<size_t>(q->L * q->rows * per_row);
  *sf_bytes = static_cast<size_t>(q->L * cdiv(q->rows, 128) * cdiv(q->cols / q->sf_vec_size, 4) * 512);
  return BSG_OK;
}

bsg_status bsg_quantize(const bsg_quant_problem* q, const void* X, void* codes, void* sf,
                        void* stream) {
  const bsg_status st = bsg_quant_check(q);
  if (st != BSG_OK) return st;
  if (!X || !codes || !sf) return BSG_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(codes) || !aligned16(sf)) return BSG_ERR_ALIGNMENT;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return BSG_ERR_CUDA;
  }
  int sms;
  {
    std::lock_guard<std::mutex> lock(g_dev_mu);
    if (g_dev_sms[dev] == 0) {
      int major = 0, minor = 0, n = 0;
      if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return BSG_ERR_CUDA;
      }
      g_dev_sms[dev] = (major == 10 && minor == 3) ? n : -1;
    }
    sms = g_dev_sms[dev];
  }
  if (sms < 0) return BSG_ERR_ARCH;
  if (q->direction == BSG_QUANT_COLWISE) return launch_colwise(q, X, codes, sf, stream, dev, sms);
  QParams p;
  std::memset(&p, 0, sizeof(p));
  const int in_bf16 = q->in_dtype == BSG_BF16 ? 1 : 0;
  const int elems = in_bf16 ? 8 : 4;
  p.x = static_cast<const uint8_t*>(X);
  p.codes = static_cast<uint8_t*>(codes);
  p.sf = static_cast<uint8_t*>(sf);
  p.row_in_bytes = q->cols * (in_bf16 ? 2 : 4);
  p.row_code_bytes = q->out_dtype == BSG_E2M1 ? q->cols / 2 : q->cols;
  p.rows = static_cast<uint32_t>(q->rows);
  p.cols = static_cast<uint32_t>(q->cols);
  p.L = static_cast<uint32_t>(q->L);
  p.chunks_per_row = static_cast<uint32_t>(q->cols / elems);
  const int64_t upr = cdiv(p.chunks_per_row, int64_t(kThreads) * unroll_of(in_bf16));
  const int64_t units = q->L * q->rows * upr;
  if (units > (int64_t(1) << 31) - 1) return BSG_ERR_INVALID_ARG;
  p.num_units = static_cast<uint32_t>(units);
  p.upr = make_fastdiv(static_cast<uint32_t>(upr));
  p.rows_div = make_fastdiv(p.rows);
  p.nblk = static_cast<uint32_t>(q->cols / q->sf_vec_size);
  p.t_r = static_cast<uint32_t>(cdiv(q->rows, 128));
  p.t_k = static_cast<uint32_t>(cdiv(p.nblk, 4));
  const int out = q->out_dtype == BSG_E4M3 ? kOutE4M3 : (q->out_dtype == BSG_E5M2 ? kOutE5M2 : kOutE2M1);
  const void* fn = pick_kernel(in_bf16, out, q->sf_vec_size);
  // one full wave of resident CTAs (as many per SM as registers allow, at
  // most 8), each striding over units: no partial second wave
  int occ;
  {
    std::lock_guard<std::mutex> lock(g_dev_mu);
    int& slot = g_dev_occ[dev][variant_of(in_bf16, out, q->sf_vec_size)];
    if (slot == 0) {
      int n = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kThreads, 0) != cudaSuccess) {
        cudaGetLastError();
        return BSG_ERR_CUDA;
      }
      slot = n < 1 ? 1 : (n > 8 ? 8 : n);
    }
    occ = slot;
  }
  const int64_t want = static_cast<int64_t>(sms) * occ;
  const int64_t extra = static_cast<int64_t>(p.L) * (p.t_k + p.t_r);
  int64_t grid = p.num_units > extra ? p.num_units : extra;
  if (grid > want) grid = want;
  if (grid < 1) grid = 1;
  void* args[1] = {&p};
  if (cudaLaunchKernel(fn, dim3(static_cast<unsigned>(grid)), dim3(kThreads), args, 0,
                       static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return BSG_ERR_CUDA;
  }
  return BSG_OK;
}

}  // extern "C"
