// Shared-memory layout of the decode attention kernel (one CTA), shared by the
// kernel, its launcher and a CPU test that checks every region's alignment for
// every batch size the kernel takes.
#pragma once

#include <cstdint>

#ifndef __CUDACC__
#define PKV_HD
#else
#define PKV_HD __host__ __device__
#endif

namespace pkv {

struct SmemLayout {
  // byte offsets from the 1024-byte aligned base; total includes the alignment slack
  uint32_t tiles, q, bars, ids, ctx, pre, prew, scratch, total;
};

// Alignment each region needs (bytes): TMA boxes of 128-byte swizzled rows land on
// 1024-byte boundaries, bulk copies of query rows need 16, mbarriers 8, everything
// else (cp.async words, schedule words) 4.
constexpr uint32_t kAlignTiles = 1024, kAlignQ = 16, kAlignBars = 8, kAlignWord = 4;

PKV_HD inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) & ~(a - 1); }

// stage_bytes: K and V tile of one stage; q_stride: per-stage query slot (a multiple
// of 128, or 0); S: sequences; nw: warps of the CTA.
PKV_HD inline SmemLayout smem_layout(int stage_bytes, int stages, int q_stride, int S, int nw) {
  SmemLayout L;
  uint32_t off = 0;
  L.tiles = off;
  off += nw * stages * stage_bytes;
  L.q = off;
  off += nw * stages * q_stride;
  off = align_up(off, 16);
  L.bars = off;
  off += nw * stages * 8;
  L.ids = off;
  off += nw * 128 * 4;  // two windows of 32 steps, up to 2 block ids per step
  L.ctx = off;
  off += S * 4;
  L.pre = off;
  off += (S + 1) * 4;
  L.prew = off;
  off += (S + 1) * 4;
  off = align_up(off, 16);
  L.scratch = off;
  off += 2 * 32 * 4;
  L.total = off + 1024;  // slack for aligning the tiles to 1024 B
  return L;
}

// True when every region of L starts on the boundary it needs (stage_bytes and
// q_stride as passed to smem_layout).
PKV_HD inline bool smem_layout_aligned(const SmemLayout& L, int stage_bytes, int q_stride) {
  return L.tiles % kAlignTiles == 0 && stage_bytes % kAlignTiles == 0 && L.q % kAlignQ == 0 &&
         q_stride % kAlignQ == 0 && L.bars % kAlignBars == 0 && L.ids % kAlignWord == 0 &&
         L.ctx % kAlignWord == 0 && L.pre % kAlignWord == 0 &&
         L.prew % kAlignWord == 0 && L.scratch % kAlignWord == 0;
}

}  // namespace pkv
