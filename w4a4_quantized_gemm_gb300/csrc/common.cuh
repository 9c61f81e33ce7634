// Shared definitions of the W4A4 library: buffer layouts (see include/w4a4.h
// for the byte-level description), launch checks, and small device helpers.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "../../include/w4a4.h"

namespace w4a4 {

constexpr int kGroup = 64;    // quantisation group along K
constexpr int kTileM = 128;   // rows per activation-workspace tile

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Packed weight buffer sections (byte offsets).
struct PackedLayout {
    size_t qW, sW, Ld, Lu, total;
};
__host__ __device__ inline PackedLayout packed_layout(int N, int K, int r) {
    PackedLayout L;
    size_t G = size_t(K) / kGroup;
    L.Ld = 0;  // first, so that the activation kernel can find it without N
    L.qW = align256(size_t(K) * size_t(r) * 2);
    L.sW = align256(L.qW + G * size_t(N) * 32);
    L.Lu = align256(L.sW + G * size_t(N) * 2);
    L.total = align256(L.Lu + size_t(r) * size_t(N) * 2);
    return L;
}

// Activation workspace sections (byte offsets).
// Stream-K hand-over area of the tcgen05 GEMM: one 64 KB slot of fp32 partial
// sums per CTA (16 epilogue warps x 4 KB) and one ready counter per (CTA, warp)
// (32 once every lane of the warp has released its part).
constexpr int kStreamKSlots = 160;      // CTAs of a stream-K launch at most
constexpr int kStreamKWarps = 16;
constexpr size_t kStreamKSlotBytes = size_t(kStreamKWarps) * 32 * 32 * 4;
constexpr int kStreamKMinM = 33;        // the area is sized in for M >= this

struct ActLayout {
    size_t qA, sS, La, flags, total;  // total: what every call needs
    size_t part, full;                // optional stream-K partial slots; full: with them
    int MT;
};
__host__ __device__ inline ActLayout act_layout(int M, int K, int r) {
    ActLayout L;
    L.MT = (M + kTileM - 1) / kTileM;
    size_t G = size_t(K) / kGroup;
    L.qA = 0;
    L.sS = align256(size_t(L.MT) * G * 2 * kTileM * 32);
    L.La = align256(L.sS + size_t(L.MT) * G * kTileM * 8);
    L.flags = align256(L.La + size_t(L.MT) * size_t(r / 16) * kTileM * 32);
    L.total = align256(L.flags + size_t(kStreamKSlots) * kStreamKWarps * 4);
    L.part = L.total;
    L.full = M >= kStreamKMinM ? L.part + size_t(kStreamKSlots) * kStreamKSlotBytes : L.total;
    return L;
}

// Fused gate|up weights packed for the SiLU(gate) * up epilogue (I gate rows,
// then I up rows; I % 16 == 0): in every 128-row tile t, each 32-row slice s
// holds 16 gate rows and then the 16 up rows of the same outputs, so that one
// epilogue thread finds both factors of an output among its 32 columns.
// Original row of packed row p: j = 64 t + 16 s + p % 16, gate j or up I + j.
__host__ __device__ inline int gate_up_row(int p, int I) {
    const int t = p >> 7, s = (p >> 5) & 3, w = p & 31;
    const int j = 64 * t + 16 * s + (w & 15);
    return w < 16 ? j : I + j;
}

// Physical 16-byte chunk of logical chunk c (0/1) in 32-byte row `row` of a
// 32-byte-swizzled plane (the tcgen05 SWIZZLE_32B pattern: address bit 4 ^= bit 7).
__host__ __device__ inline int swz32(int row, int c) { return c ^ ((row >> 2) & 1); }

// ---- offset-binary nibble -> FP8 E4M3 expansion ---------------------------
// Nibble u in [0, 15] stores code c = u - 8.  The tensor core multiplies the
// E4M3 encodings of u (exact: every integer 0..15 is an E4M3 value), so the
// per-group product is sum(cA * (cW + 8)) = P + 8 * SA, corrected in the
// epilogue.  Two byte permutes select from the 8-entry halves of the table
// E4M3(0..15): the permute's sign-fill mode turns the half not selected into
// 0x00 because every table entry is non-negative.
constexpr uint32_t kE4m3Lo0 = 0x44403800u;  // E4M3 of 0,1,2,3
constexpr uint32_t kE4m3Lo1 = 0x4E4C4A48u;  // 4,5,6,7
constexpr uint32_t kE4m3Hi0 = 0x53525150u;  // 8,9,10,11
constexpr uint32_t kE4m3Hi1 = 0x57565554u;  // 12,13,14,15

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;\n" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// The 4 nibbles in the low 16 bits of `w` -> 4 E4M3 bytes (byte i <- nibble i).
// prmt's default mode: selector bits 0-2 pick a byte, bit 3 set replicates
// that byte's sign bit (0 here) instead of copying it.
__device__ __forceinline__ uint32_t expand4(uint32_t w) {
    return prmt(kE4m3Lo0, kE4m3Lo1, w) | prmt(kE4m3Hi0, kE4m3Hi1, w ^ 0x8888u);
}

// The 8 nibbles of `w` (nibble i at bits 4i) -> 8 bytes holding the nibbles
// themselves: a = nibbles 0-3, b = nibbles 4-7 (byte i <- nibble i, the order
// of expand4).  Read as FP8 E4M3, the byte 0x0u is u * 2^-9 exactly for every
// u in [0, 15]: the subnormals (exponent field 0) are m * 2^-9 for m = 0..7
// and the first normal binade (exponent field 1) continues with (8 + m) * 2^-9.
// So the MMA sees the offset codes scaled by 2^-9 (still exact: every product
// and partial sum of a group is a multiple of 2^-9 below 2^4), and the epilogue
// multiplies by 2^9.  Five instructions for 8 nibbles instead of nine.
__device__ __forceinline__ void expand8(uint32_t w, uint32_t& a, uint32_t& b) {
    const uint32_t lo = w & 0x0F0F0F0Fu;         // nibbles 0, 2, 4, 6
    const uint32_t hi = (w >> 4) & 0x0F0F0F0Fu;  // nibbles 1, 3, 5, 7
    a = prmt(lo, hi, 0x5140u);
    b = prmt(lo, hi, 0x7362u);
}
constexpr float kExpand8Scale = 512.f;  // 2^9: the MMA product of expand8 bytes times this is the integer product

// FP8 E4M3 encoding of an integer c in [-8, 8] (exact): sign | exponent | mantissa.
__host__ __device__ __forceinline__ uint32_t e4m3_of_int(int c) {
    uint32_t s = c < 0 ? 0x80u : 0u;
    int a = c < 0 ? -c : c;
    if (a == 0) return 0u;
    int e = (a >= 8) ? 3 : (a >= 4) ? 2 : (a >= 2) ? 1 : 0;  // floor(log2 a)
    uint32_t m = (uint32_t(a) << (3 - e)) & 7u;
    return s | (uint32_t(e + 7) << 3) | m;
}

// Decode an E4M3 byte holding an integer in [-16, 16] (debug paths only).
__host__ __device__ __forceinline__ int int_of_e4m3(uint32_t b) {
    int s = (b >> 7) & 1, e = (b >> 3) & 15, m = b & 7;
    if (e == 0) return 0;
    int v = (e >= 10) ? ((8 + m) << (e - 10)) : ((8 + m) >> (10 - e));
    return s ? -v : v;
}

// ---- legacy warp-level MMA fragments (used by the small-M kernel and the
// LoRA-down of the activation kernel) ---------------------------------------
__device__ __forceinline__ void mma_e4m3_16832(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(smem)), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ uint2 ldg_nc_v2(const void* p) {
    uint2 v;
    asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];\n" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
// Programmatic dependent launch.  pdl_wait: block until the grids this one
// depends on have completed and their writes are visible (a no-op when the
// launch has no such dependency); every kernel calls it before its first
// access to global memory, so no read or write can race with the previous
// kernel in the stream.  pdl_launch_dependents: allow the next grid to be
// scheduled now, so that its launch overlaps this grid's work.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// Read-only 16-byte load that does not allocate in L1 (data read once).
__device__ __forceinline__ uint4 ldg_stream_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

}  // namespace w4a4

// ---- host-side launch helpers (implemented in api.cu) ----------------------
namespace w4a4 {
void set_dispatch(const char* fmt, ...);
w4a4_status launch_status();  // maps cudaGetLastError() to a status
int device_sm_count();        // multiprocessors of the current device (cached)
// Appends the programmatic-stream-serialisation attribute (the launch may
// overlap the previous kernel in the stream, which its pdl_wait orders) unless
// W4A4_PDL=0 is set in the environment; returns the new attribute count.
unsigned add_pdl_attr(cudaLaunchAttribute* attrs, unsigned n);
bool tc_stream_k_enabled();
w4a4_status tc_read_and_clear_status();      // bounded-wait status of the tcgen05 kernel
w4a4_status smallm_read_and_clear_status();  // bounded-wait status of the small-M kernel
w4a4_status w4a16_read_and_clear_status();   // bounded-wait status of the W4A16 kernel
w4a4_status smtc_read_and_clear_status();    // bounded-wait status of the tcgen05 small-M kernel
w4a4_status q_read_and_clear_status();       // bounded-wait status of the activation kernel
w4a4_status fused_read_and_clear_status();   // bounded-wait status of the fused small-M linear
}  // namespace w4a4
