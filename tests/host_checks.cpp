// host_checks.cpp — the C ABI's host side under AddressSanitizer and
// UndefinedBehaviorSanitizer, without a GPU: status strings, cache
// accounting, the launch planning behind every workspace-size query over a
// grid of shapes (LRKV_SM_COUNT set by the caller, so no device is asked),
// and the argument checks of every compute entry point (each must reject a
// null or malformed argument before it touches the device).  Exit status 0
// when every expectation holds; each failure is printed.
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <initializer_list>

#include "lrkv.h"

static int g_fail = 0;

#define EXPECT(cond)                                                    \
  do {                                                                  \
    if (!(cond)) {                                                      \
      std::fprintf(stderr, "%s:%d: expected %s\n", __FILE__, __LINE__, #cond); \
      ++g_fail;                                                         \
    }                                                                   \
  } while (0)

static lrkv_dims dims(int B, int H, int dh, int r, int L, lrkv_dtype t) {
  lrkv_dims d;
  std::memset(&d, 0, sizeof(d));
  d.batch = B;
  d.heads = H;
  d.head_dim = dh;
  d.rank = r;
  d.max_len = L;
  d.dtype = t;
  d.scale = 0.f;
  return d;
}

int main() {
  // ---- strings and accounting ------------------------------------------------
  EXPECT(lrkv_abi_version() > 0);
  for (int s = -3; s < 10; ++s) EXPECT(lrkv_status_string(static_cast<lrkv_status>(s)) != nullptr);
  EXPECT(std::strcmp(lrkv_status_string(LRKV_OK), "LRKV_OK") == 0);
  EXPECT(lrkv_cache_elems_per_token(32, 128, 48) == 2u * (128u + 32u * 48u));
  EXPECT(lrkv_cache_elems_per_token(-1, 128, 48) == 0u);

  // ---- planning: decode workspace sizes over a grid of shapes -------------------
  const int Bs[] = {1, 3, 8, 32, 4096};
  const int Hs[] = {1, 4, 16, 18, 32, 64};
  const int dhs[] = {16, 64, 128};
  const int rs[] = {0, 4, 8, 12, 16, 28, 48, 56, 64};
  const int Ls[] = {1, 64, 300, 4096, 65536};
  int planned = 0;
  for (lrkv_dtype t : {LRKV_BF16, LRKV_F32})
    for (int B : Bs)
      for (int H : Hs)
        for (int dh : dhs)
          for (int r : rs)
            for (int L : Ls) {
              const lrkv_dims d = dims(B, H, dh, r, L, t);
              size_t n = 0;
              const lrkv_status st = lrkv_decode_workspace_size(&d, &n);
              EXPECT(st == LRKV_OK || st == LRKV_ERR_UNSUPPORTED);
              if (st == LRKV_OK) {
                EXPECT(n >= 16);
                ++planned;
              }
              size_t nr = 0;
              const lrkv_status sr = lrkv_decode_rope_workspace_size(&d, &nr);
              EXPECT(sr == LRKV_OK || sr == LRKV_ERR_UNSUPPORTED || sr == LRKV_ERR_INVALID_ARG);
              size_t np = 0;
              const lrkv_status sp = lrkv_prefill_workspace_size(&d, L, &np);
              EXPECT(sp == LRKV_OK || sp == LRKV_ERR_UNSUPPORTED || sp == LRKV_ERR_INVALID_ARG);
            }
  EXPECT(planned > 100);
  for (int Hkv : {1, 2, 4, 8, 32})
    for (int d : {64, 128}) {
      lrkv_dense_dims dd;
      std::memset(&dd, 0, sizeof(dd));
      dd.batch = 4; dd.heads = 32; dd.kv_heads = Hkv; dd.head_dim = d; dd.max_len = 4096;
      size_t n = 0;
      const lrkv_status st = lrkv_dense_decode_workspace_size(&dd, &n);
      EXPECT(st == LRKV_OK || st == LRKV_ERR_UNSUPPORTED);
    }
  {
    lrkv_mla_dims md;
    std::memset(&md, 0, sizeof(md));
    md.batch = 4; md.heads = 32; md.head_dim = 128; md.latent_dim = 512; md.max_len = 4096;
    size_t n = 0;
    const lrkv_status st = lrkv_mla_decode_workspace_size(&md, &n);
    EXPECT(st == LRKV_OK || st == LRKV_ERR_UNSUPPORTED);
  }

  // ---- malformed arguments: rejected before the device is touched --------------
  const lrkv_dims good = dims(2, 16, 64, 28, 256, LRKV_BF16);
  lrkv_dims bad = good;
  bad.batch = 0;
  size_t n = 0;
  EXPECT(lrkv_decode_workspace_size(nullptr, &n) == LRKV_ERR_INVALID_ARG);
  EXPECT(lrkv_decode_workspace_size(&good, nullptr) == LRKV_ERR_INVALID_ARG);
  EXPECT(lrkv_decode_workspace_size(&bad, &n) == LRKV_ERR_INVALID_ARG);
  lrkv_dims nan_scale = good;
  std::memcpy(&nan_scale.scale, "\xff\xff\xff\x7f", 4);
  EXPECT(lrkv_decode_workspace_size(&nan_scale, &n) == LRKV_ERR_INVALID_ARG);
  // a fake, aligned, never dereferenced device address for the other operands
  void* p = reinterpret_cast<void*>(static_cast<uintptr_t>(1) << 20);
  float* f = static_cast<float*>(p);
  const int32_t* i32 = static_cast<const int32_t*>(p);
  EXPECT(lrkv_decode(nullptr, p, p, p, p, p, p, p, i32, f, f, p, 1 << 20, nullptr) == LRKV_ERR_INVALID_ARG);
  EXPECT(lrkv_decode(&good, nullptr, p, p, p, p, p, p, i32, f, f, p, 1 << 20, nullptr) == LRKV_ERR_INVALID_ARG);
  EXPECT(lrkv_decode(&good, p, p, p, p, p, p, p, nullptr, f, f, p, 1 << 20, nullptr) == LRKV_ERR_INVALID_ARG);
  EXPECT(lrkv_decode(&good, p, p, p, p, p, p, p, i32, f, f, nullptr, 0, nullptr) == LRKV_ERR_WORKSPACE);
  void* odd = reinterpret_cast<void*>((static_cast<uintptr_t>(1) << 20) + 8);
  EXPECT(lrkv_decode(&good, odd, p, p, p, p, p, p, i32, f, f, p, 1 << 20, nullptr) == LRKV_ERR_INVALID_ARG);
  EXPECT(lrkv_decode_normed(&good, p, p, p, p, p, p, p, nullptr, i32, f, f, p, 1 << 20, nullptr) ==
         LRKV_ERR_INVALID_ARG);
  EXPECT(lrkv_decode_paged(&good, 64, 8, nullptr, p, p, p, p, p, p, p, i32, f, f, p, 1 << 20, nullptr) ==
         LRKV_ERR_INVALID_ARG);
  EXPECT(lrkv_decode_paged(&good, 48, 8, i32, p, p, p, p, p, p, p, i32, f, f, p, 1 << 20, nullptr) ==
         LRKV_ERR_INVALID_ARG);  // page size not a power of two
  EXPECT(lrkv_key_scales(&good, 1e-6f, 16, nullptr, p, p, i32, f, nullptr) == LRKV_ERR_INVALID_ARG);
  EXPECT(lrkv_append(nullptr, 256, 16, p, p, p, p, p, i32, p, p, p, p, p, 16, nullptr) == LRKV_ERR_INVALID_ARG);
  EXPECT(lrkv_append(&good, 256, 16, nullptr, p, p, p, p, i32, p, p, p, p, p, 16, nullptr) ==
         LRKV_ERR_INVALID_ARG);
  EXPECT(lrkv_append(&good, 256, 16, p, p, p, p, p, i32, p, p, p, p, nullptr, 0, nullptr) ==
         LRKV_ERR_WORKSPACE);
  const lrkv_dims pf = dims(2, 4, 128, 64, 256, LRKV_BF16);
  EXPECT(lrkv_prefill(&pf, 64, nullptr, p, p, p, p, p, p, i32, f, f, p, 16, nullptr) == LRKV_ERR_INVALID_ARG);
  EXPECT(lrkv_prefill(&pf, 64, p, p, p, p, p, p, p, i32, f, f, p, 8, nullptr) == LRKV_ERR_WORKSPACE);
  EXPECT(lrkv_prefill(&pf, 512, p, p, p, p, p, p, p, i32, f, f, p, 16, nullptr) != LRKV_OK);  // q_len > max_len
  EXPECT(lrkv_decode_step(&good, 256, nullptr, p, p, p, p, p, p, p, p, p, p, p, i32, f, f, p, 1 << 20,
                          nullptr) == LRKV_ERR_INVALID_ARG);
  EXPECT(lrkv_rope_table(0, 64, 10000.f, f, nullptr) == LRKV_ERR_INVALID_ARG);
  EXPECT(lrkv_read_device_status(nullptr, nullptr, nullptr) == LRKV_ERR_INVALID_ARG);
  EXPECT(lrkv_read_static_scratch_status(nullptr, nullptr) == LRKV_ERR_INVALID_ARG);

  if (g_fail) std::fprintf(stderr, "%d expectation(s) failed\n", g_fail);
  else std::printf("host checks ok: %d decode plans\n", planned);
  return g_fail ? 1 : 0;
}
