// Route-count history file (".coli_usage"), host side.
//
// Page: "colibrì 路由遥测全解析.coli_usage专家历史、ROUTE_TRACE追踪流与route_trace.h统一格式",
// §历史文件 (text records of exactly three numeric fields; the -1 geometry and
// -2 version / engine-hash header records; nonzero counts only; temporary file
// plus rename; an empty history is a 0-byte file), §编辑格式前必须知道的两个后果
// (the 32-bit hash sits in the third field), §可信读取 (a trusted read relaxes
// the engine identity only, never the geometry or the format version), and the
// COLI_USAGE_DECAY description (a per-save multiplier in (0, 1], rounding that
// keeps count-1 experts).
#include <errno.h>
#include <limits.h>
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <vector>

#include "coli.h"

namespace {

constexpr int kUsageVersion = 1;
constexpr unsigned char kDenseMagic[4] = {'I', 'K', 'U', '1'};   // dense binary layout
constexpr size_t kMaxPath = 4096;

struct Record {
  long long l, e;
  unsigned long long c;
};

// Reads the next "a b c" record: three whitespace-separated decimal integers.
// Returns false at the end of the file or at anything that is not such a
// record (the record stream ends there, as with a scanf loop).
bool next_record(FILE *f, Record *r) {
  long long a, b;
  unsigned long long c;
  if (fscanf(f, "%lld %lld %llu", &a, &b, &c) != 3) return false;
  r->l = a;
  r->e = b;
  r->c = c;
  return true;
}

uint32_t decayed(uint32_t c, float decay) {
  if (c == 0 || !(decay > 0.0f && decay < 1.0f)) return c;
  const double v = floor((double)c * (double)decay + 0.5);
  return v < 1.0 ? 1u : (uint32_t)v;
}

}  // namespace

extern "C" {

uint32_t coli_usage_engine_id(const char *engine) {
  uint32_t h = 2166136261u;
  for (const unsigned char *p = (const unsigned char *)(engine ? engine : ""); *p; ++p) {
    h ^= *p;
    h *= 16777619u;
  }
  return h;
}

int coli_usage_save(const char *path, const uint32_t *counts, int32_t n_layers, int32_t n_experts,
                    const char *engine, float decay) {
  if (!path || !counts || !engine || n_layers <= 0 || n_experts <= 0) return COLI_EINVAL;
  char tmp[kMaxPath];
  const int n = snprintf(tmp, sizeof(tmp), "%s.tmp", path);
  if (n < 0 || (size_t)n >= sizeof(tmp)) return COLI_EINVAL;   // nothing touched yet
  const size_t total = (size_t)n_layers * (size_t)n_experts;
  bool any = false;
  for (size_t i = 0; i < total && !any; ++i) any = decayed(counts[i], decay) != 0;
  FILE *f = fopen(tmp, "wb");
  if (!f) return COLI_EIO;
  bool ok = true;
  if (any) {
    ok = fprintf(f, "-1 %d %d\n-2 %d %u\n", (int)n_layers, (int)n_experts, kUsageVersion,
                 coli_usage_engine_id(engine)) > 0;
    for (int32_t l = 0; l < n_layers && ok; ++l)
      for (int32_t e = 0; e < n_experts && ok; ++e) {
        const uint32_t c = decayed(counts[(size_t)l * n_experts + e], decay);
        if (c) ok = fprintf(f, "%d %d %u\n", (int)l, (int)e, c) > 0;
      }
  }
  ok = (fflush(f) == 0) && ok;
  ok = (fclose(f) == 0) && ok;
  if (ok) ok = rename(tmp, path) == 0;
  if (!ok) {
    remove(tmp);
    return COLI_EIO;
  }
  return COLI_OK;
}

int coli_usage_load(const char *path, uint32_t *counts, int32_t n_layers, int32_t n_experts,
                    const char *engine, int trusted, int64_t *n_records) {
  if (n_records) *n_records = 0;
  if (!path || !counts || !engine || n_layers <= 0 || n_experts <= 0) return COLI_EINVAL;
  FILE *f = fopen(path, "rb");
  if (!f) return COLI_EIO;
  unsigned char head[4] = {0, 0, 0, 0};
  const size_t got = fread(head, 1, 4, f);
  if (got == 4 && memcmp(head, kDenseMagic, 4) == 0) {
    fclose(f);
    return COLI_EREFUSED;   // another engine's dense binary history
  }
  rewind(f);
  // the whole file is checked before any count is added
  std::vector<Record> data;
  const uint32_t me = coli_usage_engine_id(engine);
  int status = COLI_OK;
  Record r;
  while (status == COLI_OK && next_record(f, &r)) {
    if (r.l >= 0) {
      if (r.l < n_layers && r.e >= 0 && r.e < n_experts && r.c <= UINT_MAX) data.push_back(r);
      continue;   // outside the geometry: discarded, not counted
    }
    if (r.l == -1) {
      if (r.e != n_layers || r.c != (unsigned long long)n_experts) status = COLI_EREFUSED;
    } else if (r.l == -2) {
      if (r.e > kUsageVersion) status = COLI_EREFUSED;
      else if (r.c != (unsigned long long)me && !trusted) status = COLI_EREFUSED;
    }
    // other negative kinds: later header records, skipped
  }
  fclose(f);
  if (status != COLI_OK) return status;
  for (const Record &d : data) {
    uint32_t &dst = counts[(size_t)d.l * n_experts + d.e];
    const unsigned long long v = (unsigned long long)dst + d.c;
    dst = v > UINT_MAX ? UINT_MAX : (uint32_t)v;
  }
  if (n_records) *n_records = (int64_t)data.size();
  return COLI_OK;
}

}  // extern "C"
