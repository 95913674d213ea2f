// io.cu -- int32 token files (gpt2_tokens_*).
//
// InfoQ's account of llm.c, section on preparing the data: each split is
// written as a .bin file holding the raw bytes of int32 GPT-2 token ids,
// which the trainer reads to feed its forward pass.  This reader keeps the
// whole file in host memory and serves next-token batches from a cursor;
// the semantics are documented with the declarations in gpt2.h.  Host code
// only: no kernel runs here.
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "../../include/gpt2.h"
#include "kernels.h"

struct gpt2_tokens {
  std::vector<int32_t> s;
  int64_t pos = 0;
};

extern "C" {

int gpt2_tokens_open(const char* path, gpt2_tokens** out) {
  if (!path || !out) {
    set_global_error("gpt2_tokens_open: NULL argument");
    return GPT2_ERR_ARG;
  }
  *out = nullptr;
  FILE* f = std::fopen(path, "rb");
  if (!f) {
    set_global_error((std::string("gpt2_tokens_open: cannot open ") + path).c_str());
    return GPT2_ERR_IO;
  }
  std::fseek(f, 0, SEEK_END);
  const long bytes = std::ftell(f);
  std::fseek(f, 0, SEEK_SET);
  if (bytes < 0) {
    std::fclose(f);
    set_global_error("gpt2_tokens_open: cannot size the file");
    return GPT2_ERR_IO;
  }
  if (bytes % 4 != 0) {
    std::fclose(f);
    set_global_error("gpt2_tokens_open: file size is not a multiple of 4 bytes");
    return GPT2_ERR_ARG;
  }
  gpt2_tokens* d = new (std::nothrow) gpt2_tokens;
  if (!d) {
    std::fclose(f);
    set_global_error("gpt2_tokens_open: out of host memory");
    return GPT2_ERR_OOM;
  }
  try {
    d->s.resize((size_t)(bytes / 4));
  } catch (...) {
    delete d;
    std::fclose(f);
    set_global_error("gpt2_tokens_open: out of host memory");
    return GPT2_ERR_OOM;
  }
  const size_t got = std::fread(d->s.data(), sizeof(int32_t), d->s.size(), f);
  std::fclose(f);
  if (got != d->s.size()) {
    delete d;
    set_global_error("gpt2_tokens_open: short read");
    return GPT2_ERR_IO;
  }
  *out = d;
  return GPT2_OK;
}

int gpt2_tokens_count(const gpt2_tokens* d, int64_t* n) {
  if (!d || !n) return GPT2_ERR_ARG;
  *n = (int64_t)d->s.size();
  return GPT2_OK;
}

int gpt2_tokens_next_batch(gpt2_tokens* d, int32_t B, int32_t T, int32_t* tokens, int32_t* targets) {
  if (!d || !tokens || !targets || B < 1 || T < 1) {
    set_global_error("gpt2_tokens_next_batch: NULL argument or B, T < 1");
    return GPT2_ERR_ARG;
  }
  const int64_t bt = (int64_t)B * T, n = (int64_t)d->s.size();
  if (bt + 1 > n) {
    set_global_error("gpt2_tokens_next_batch: the file holds fewer than B*T+1 tokens");
    return GPT2_ERR_ARG;
  }
  if (d->pos + bt + 1 > n) d->pos = 0;  // start over
  std::memcpy(tokens, d->s.data() + d->pos, (size_t)bt * sizeof(int32_t));
  std::memcpy(targets, d->s.data() + d->pos + 1, (size_t)bt * sizeof(int32_t));
  d->pos += bt;
  return GPT2_OK;
}

int gpt2_tokens_reset(gpt2_tokens* d) {
  if (!d) return GPT2_ERR_ARG;
  d->pos = 0;
  return GPT2_OK;
}

void gpt2_tokens_close(gpt2_tokens* d) { delete d; }

}  // extern "C"
