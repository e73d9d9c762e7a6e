// Device helpers shared by the kernels of the W2-g128 folded-Hadamard layer.
// sm_103a only: mbarrier / bulk-copy / tcgen05 PTX is written inline.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/tb.h"

#define TB_DEVI __device__ __forceinline__

// Upper bound of every spin on an mbarrier, in nanoseconds of %globaltimer.
// A wait that runs out records TB_DEV_TIMEOUT and the kernel winds down.
#ifndef TB_WAIT_NS
#define TB_WAIT_NS 2000000000ull
#endif

namespace tb {

constexpr int kGroup = 128;        // weights per scale/bias group
constexpr int kCodesPerWord = 16;  // 2-bit codes per uint32
constexpr int kBlock = 1024;       // Hadamard block
constexpr float kInvSqrtBlock = 1.0f / 32.0f;

// ---------------------------------------------------------------- addresses
TB_DEVI uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

TB_DEVI uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// gpu-scope release/acquire fence: orders this thread's earlier accesses (and, through a
// preceding warp barrier, its warp's) before its later ones for every thread on the GPU,
// without the cost of a sequentially consistent fence
TB_DEVI void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// gpu-scope acquire load of a 32-bit counter in global memory
TB_DEVI uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

TB_DEVI void set_status(int32_t* st, int bits) {
  if (st) atomicOr(st, bits);
}

// ---------------------------------------------------------------- mbarrier
TB_DEVI void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

// make barrier initialisation visible to the async proxy (bulk copies, tcgen05)
TB_DEVI void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

TB_DEVI void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

TB_DEVI void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

TB_DEVI void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

TB_DEVI bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.  Returns false
// when TB_WAIT_NS elapsed first.
TB_DEVI bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > TB_WAIT_NS) return false;
  }
}

// ---------------------------------------------------------------- bulk copies
// 1-D bulk copy global -> shared, completion counted in bytes on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
TB_DEVI void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Same with an L2 evict-first policy: for data read exactly once (weights).
TB_DEVI uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

TB_DEVI void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                           uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// ---------------------------------------------------------------- explicit shared-memory access
// (32-bit shared addresses: no generic-address resolution on the hot path)
TB_DEVI uint4 ld_shared_v4(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
TB_DEVI uint2 ld_shared_v2(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
TB_DEVI float2 ld_shared_f2(uint32_t a) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0,%1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a));
  return v;
}
TB_DEVI float ld_shared_f(uint32_t a) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
  return v;
}
TB_DEVI float ld_shared_half(uint32_t a) {
  unsigned short h;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h) : "r"(a));
  return __half2float(__ushort_as_half(h));
}
TB_DEVI void st_shared_f(uint32_t a, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}
TB_DEVI void red_shared_add(uint32_t a, float v) {
  asm volatile("red.shared.add.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}

// ---------------------------------------------------------------- small ALU helpers
TB_DEVI uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;  // (a & b) | c
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

TB_DEVI uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

TB_DEVI float half_bits_to_float(uint16_t b) { return __half2float(__ushort_as_half(b)); }

// ---------------------------------------------------------------- warp FWHT
// 32 values per lane; two layouts of a 1024-block:
//   layout A: v[r] is element lane*32 + r
//   layout B: v[j] is element j*32 + lane
// The transform's 10 butterfly stages commute, so the stages over the
// in-register index bits run in whichever layout is current.

// the five butterfly stages over the register index (bits 0..4 of it)
TB_DEVI void butterfly32(float (&v)[32]) {
#pragma unroll
  for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if ((i & h) == 0) {
        const float a = v[i], b = v[i + h];
        v[i] = a + b;
        v[i + h] = a - b;
      }
    }
  }
}

// layout B -> layout A through a padded 32x33 float scratch owned by the warp
TB_DEVI void transpose_b_to_a(float (&v)[32], float* scratch, int lane) {
#pragma unroll
  for (int j = 0; j < 32; ++j) scratch[j * 33 + lane] = v[j];
  __syncwarp();
#pragma unroll
  for (int r = 0; r < 32; ++r) v[r] = scratch[lane * 33 + r];
  __syncwarp();
}

// layout A -> layout B
TB_DEVI void transpose_a_to_b(float (&v)[32], float* scratch, int lane) {
#pragma unroll
  for (int r = 0; r < 32; ++r) scratch[lane * 33 + r] = v[r];
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = scratch[j * 33 + lane];
  __syncwarp();
}

// unnormalised Walsh-Hadamard transform of one 1024-block held by a warp:
// in: layout B, out: layout A
TB_DEVI void wht1024_b_to_a(float (&v)[32], float* scratch, int lane) {
  butterfly32(v);  // element bits 5..9
  transpose_b_to_a(v, scratch, lane);
  butterfly32(v);  // element bits 0..4
}

// in: layout A, out: layout B
TB_DEVI void wht1024_a_to_b(float (&v)[32], float* scratch, int lane) {
  butterfly32(v);  // element bits 0..4
  transpose_a_to_b(v, scratch, lane);
  butterfly32(v);  // element bits 5..9
}

constexpr int kWarpScratchFloats = 32 * 33;

// Unnormalised Walsh-Hadamard transform of a 1024-block in layout A without shared memory:
// five butterfly stages over the register index (element bits 0..4), then five over the
// lane index (element bits 5..9) with xor-shuffles; the result stays in layout A.
TB_DEVI void wht1024_a_shfl(float (&v)[32], int lane) {
  butterfly32(v);
#pragma unroll
  for (int h = 1; h < 32; h <<= 1) {
    const float sg = (lane & h) ? -1.0f : 1.0f;  // upper partner keeps a - b
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      const float p = __shfl_xor_sync(0xffffffffu, v[r], h);
      v[r] = fmaf(sg, v[r], p);
    }
  }
}

// Unnormalised Walsh-Hadamard transform of 512 elements held by a warp as v[e] = element
// lane*16 + e: four butterfly stages over the register index (element bits 0..3), then five
// over the lane index (bits 4..8) with xor-shuffles; the layout is kept.
TB_DEVI void wht512_a_shfl(float (&v)[16], int lane) {
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if ((i & h) == 0) {
        const float a = v[i], b = v[i + h];
        v[i] = a + b;
        v[i + h] = a - b;
      }
    }
  }
#pragma unroll
  for (int h = 1; h < 32; h <<= 1) {
    const float sg = (lane & h) ? -1.0f : 1.0f;  // upper partner keeps a - b
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const float p = __shfl_xor_sync(0xffffffffu, v[r], h);
      v[r] = fmaf(sg, v[r], p);
    }
  }
}

// Same transform through a 4 KB shared scratch owned by the warp: 32 rows of 128 bytes, the
// 16-byte chunk c of row i stored at position c ^ (i & 7).  Five stages over the register
// index (element bits 0..4); each lane writes its row as eight 16-byte chunks; each lane reads
// column `lane` (layout B); five more stages (bits 5..9); the same way back.  Row accesses
// are conflict-free per 8-lane phase, column accesses over all 32 banks; addresses are eight
// bases plus immediate offsets, so the transposes need few registers.
TB_DEVI void wht1024_a_smem(float (&v)[32], uint32_t scratch, int lane) {
  butterfly32(v);
  const uint32_t row = scratch + (uint32_t)lane * 128u;
  const uint32_t sw = (uint32_t)lane & 7u;
#pragma unroll
  for (int c = 0; c < 8; ++c)
    asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(row + 16u * ((uint32_t)c ^ sw)),
                 "f"(v[4 * c]), "f"(v[4 * c + 1]), "f"(v[4 * c + 2]), "f"(v[4 * c + 3])
                 : "memory");
  __syncwarp();
  uint32_t col[8];  // word `lane` of row j lies at col[j & 7] + 128 j
#pragma unroll
  for (int k = 0; k < 8; ++k) col[k] = scratch + 16u * (((uint32_t)lane >> 2) ^ (uint32_t)k) + 4u * ((uint32_t)lane & 3u);
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = ld_shared_f(col[j & 7] + 128u * (uint32_t)j);
  butterfly32(v);
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 32; ++j) st_shared_f(col[j & 7] + 128u * (uint32_t)j, v[j]);
  __syncwarp();
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    float4 q;
    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(q.x), "=f"(q.y), "=f"(q.z), "=f"(q.w)
                 : "r"(row + 16u * ((uint32_t)c ^ sw))
                 : "memory");
    v[4 * c] = q.x;
    v[4 * c + 1] = q.y;
    v[4 * c + 2] = q.z;
    v[4 * c + 3] = q.w;
  }
  __syncwarp();
}

// Sum of 32 values as a balanced tree (depth 5 instead of a 32-long dependent chain).
TB_DEVI float tree_sum32(const float (&v)[32]) {
  float s[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) s[i] = v[2 * i] + v[2 * i + 1];
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) s[i] = s[2 * i] + s[2 * i + 1];
  return s[0];
}

// Same transform, register-light: the five lane stages run on eight register indices at a
// time (each index is an independent chain through the five stages), so a warp keeps eight
// shuffles in flight with eight extra registers instead of serialising them when registers
// are scarce.
TB_DEVI void wht1024_a_shfl_batched(float (&v)[32], int lane) {
  butterfly32(v);
#pragma unroll
  for (int rb = 0; rb < 32; rb += 8) {
#pragma unroll
    for (int h = 1; h < 32; h <<= 1) {
      const float sg = (lane & h) ? -1.0f : 1.0f;
      float p[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) p[r] = __shfl_xor_sync(0xffffffffu, v[rb + r], h);
#pragma unroll
      for (int r = 0; r < 8; ++r) v[rb + r] = fmaf(sg, v[rb + r], p[r]);
    }
  }
}

}  // namespace tb
