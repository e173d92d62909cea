// Problem geometry shared by the host launcher and the kernels.
#pragma once

#include <stdint.h>

namespace rkv {

constexpr int kHeadDim = 128;       // d: one key row = 256 bytes of bf16
constexpr int kTileKeys = 128;      // keys per tensor-core tile (the MMA M dimension)
constexpr int kHalfBytes = 16384;   // one 64-column half of a 128x128 bf16 tile
constexpr int kTileBytes = 32768;   // a full 128x128 bf16 tile
constexpr int kBlock = 16;          // paged block size
constexpr int kMaxSeq = 8192;       // largest supported max_seq_len

struct Geom {
    int L, B, Hkv, Hq, G, w, rows; // rows = w * G query rows per KV head
    int nmax;                       // max_seq_len
    int npad;                       // score stride: round_up(nmax, 128)
    int paged;
    int max_blocks, num_blocks;
    int budget;
    float lam;
    int redundancy; // rkv_redundancy_method
    int shared_sel; // rkv_selection == RKV_SELECT_SHARED_HEADS
    int buffer;
    int trigger_at_full; // rkv_trigger == RKV_TRIGGER_BUDGET_PLUS_BUFFER
    const int32_t *seq_lens;
    const int32_t *block_table;
};

// Whether a sequence holding n tokens is compressed by this call: always
// (n <= budget is then a no-op), or, with the device-side trigger, only once it
// holds budget + buffer tokens.
__host__ __device__ inline bool triggered(const Geom &g, int n)
{
    return !g.trigger_at_full || n >= g.budget + g.buffer;
}

// Head index e = (l * B + b) * Hkv + h.
struct HeadId {
    int l, b, h;
};

__host__ __device__ inline HeadId head_id(const Geom &g, int e)
{
    HeadId id;
    id.h = e % g.Hkv;
    id.b = (e / g.Hkv) % g.B;
    id.l = e / (g.Hkv * g.B);
    return id;
}

} // namespace rkv
