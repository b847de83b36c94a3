// Runs the decompress launch planner (zvc_plan.h) on the host against a model of a GB300
// SM's limits and prints one JSON line per case, for tests/test_plan_cpu.py to check.
//
// The model: 152 SMs; per SM 65536 registers allocated per warp in units of 256, 228 KB of
// shared memory (1 KB of it reserved per CTA), at most 32 CTAs and 64 warps; at most
// 227 KB of shared memory per CTA. Registers per thread: 47, or 32 for chunks of at most
// 1024 elements (the two builds of the kernel).
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "zvc_plan.h"

using zvc::plan::Limits;
using zvc::plan::Plan;

static const Limits kGB300 = {152, 233472, 1024, 232448};

static int model_occ(uint32_t C, uint32_t k, uint32_t cap) {
  const int warps = (int)(1 + k);
  const int regs = C <= 1024 ? 32 : 47;
  const int warp_regs = (regs * 32 + 255) / 256 * 256;
  const int by_regs = 65536 / (warps * warp_regs);
  const uint64_t smem = k * zvc::plan::slot_bytes(cap, C);
  if (smem > (uint64_t)kGB300.smem_per_cta_max) return 0;
  const int by_smem = (int)(kGB300.smem_per_sm / (smem + kGB300.reserved_per_cta));
  int n = by_regs < by_smem ? by_regs : by_smem;
  if (n > 32) n = 32;
  if (n > 64 / warps) n = 64 / warps;
  return n;
}

// Compressed bytes of a single stream: header, chunk table, a mask per window, the
// non-zero words.
static uint64_t stream_bytes(uint64_t n, uint32_t C, uint64_t nnz) {
  return 32 + 8 * ((n + C - 1) / C) + 4 * ((n + 31) / 32) + 4 * nnz;
}

static void run(const char* name, uint64_t chunks, uint64_t in_bytes, uint32_t T, bool batched,
                uint32_t C) {
  auto occ = [C](uint32_t k, uint32_t cap) { return model_occ(C, k, cap); };
  Plan p;
  const bool ok = zvc::plan::decompress_plan(chunks, in_bytes, T, batched, C, kGB300, occ, &p);
  const uint32_t full = zvc::plan::full_cap_words(C);
  uint64_t mean = zvc::plan::mean_chunk_words(in_bytes, chunks, T, batched);
  if (mean > full) mean = full;
  const int o = ok ? model_occ(C, p.chunks_per_cta, p.cap_words) : 0;
  printf("{\"case\": \"%s\", \"ok\": %d, \"chunks\": %llu, \"C\": %u, \"full\": %u, "
         "\"mean\": %llu, \"cap\": %u, \"k\": %u, \"occ\": %d, \"occ1_min_cap\": %d, "
         "\"slot_bytes\": %llu}\n",
         name, ok ? 1 : 0, (unsigned long long)chunks, C, full, (unsigned long long)mean,
         p.cap_words, p.chunks_per_cta, o, model_occ(C, 1, zvc::plan::kCapMinWords),
         (unsigned long long)zvc::plan::slot_bytes(p.cap_words, C));
}

static void single(const char* name, uint64_t n, uint32_t C, double density) {
  const uint64_t nnz = (uint64_t)(density * (double)n);
  run(name, (n + C - 1) / C, stream_bytes(n, C, nnz), 1, false, C);
}

int main() {
  single("alexnet0_dense", 37171200, 4096, 1.0);
  single("alexnet0_60", 37171200, 4096, 0.6);
  single("alexnet1_45", 23887872, 4096, 0.45);
  single("alexnet4_20", 5537792, 4096, 0.2);
  single("sweep_0", 1ull << 28, 4096, 0.0);
  single("sweep_10", 1ull << 28, 4096, 0.1);
  single("sweep_50", 1ull << 28, 4096, 0.5);
  single("sweep_100", 1ull << 28, 4096, 1.0);
  single("c1024_sweep_50", 1ull << 28, 1024, 0.5);
  single("c1024_small", 200704, 1024, 0.5);
  single("c32_sweep_0", 1ull << 24, 32, 0.0);
  single("c16384_dense", 1ull << 22, 16384, 1.0);
  single("c32768_dense", 8 * 32768, 32768, 1.0);
  // a batch: 3 tensors (one empty), 16 + 8 * (T + 1) bytes of batch header and table
  {
    const uint32_t C = 4096;
    const uint64_t n[3] = {30000000, 0, 5000000};
    uint64_t S = 16 + 8 * 4, chunks = 0;
    for (int i = 0; i < 3; ++i) {
      S += stream_bytes(n[i], C, n[i] / 4);
      chunks += (n[i] + C - 1) / C;
    }
    run("batch_25", chunks, S, 3, true, C);
  }
  run("no_chunks", 0, 32, 1, false, 4096);
  run("truncated", 9075, 100, 1, false, 4096);  // smaller than its own tables
  // an occupancy query that fails: the planner reports it
  {
    Plan p;
    const bool ok = zvc::plan::decompress_plan(
        9075, 94000000, 1, false, 4096, kGB300, [](uint32_t, uint32_t) { return -1; }, &p);
    printf("{\"case\": \"occ_error\", \"ok\": %d}\n", ok ? 1 : 0);
  }
  return 0;
}
