// diag.cu -- the MLQ_DIAG=1 kernel-choice report (see diag.h).
#include "diag.h"

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cxxabi.h>
#include <mutex>
#include <string>
#include <unordered_set>

namespace mlq {

namespace {
thread_local std::string t_entry;  // "mlq_xxx shape..."
thread_local std::string t_note;   // geometry of the next launch
std::mutex g_mu;

std::string vformat(const char *fmt, va_list ap) {
  char buf[512];
  vsnprintf(buf, sizeof(buf), fmt, ap);
  return buf;
}

std::string kernel_name(const void *kern) {
  const char *name = nullptr;
  if (cudaFuncGetName(&name, kern) != cudaSuccess || name == nullptr) {
    cudaGetLastError();
    return "?";
  }
  int st = 0;
  char *dem = abi::__cxa_demangle(name, nullptr, nullptr, &st);
  std::string out = st == 0 && dem != nullptr ? dem : name;
  std::free(dem);
  // drop the parameter list: "mlq::phase_ring_kernel<0, 16>(mlq::PhaseArgs)" -> "...<0, 16>"
  const size_t p = out.find('(');
  if (p != std::string::npos) out.resize(p);
  return out;
}
}  // namespace

bool diag_on() {
  static const bool on = [] {
    const char *e = std::getenv("MLQ_DIAG");
    return e != nullptr && e[0] == '1';
  }();
  return on;
}

void diag_entry(const char *entry, const char *fmt, ...) {
  if (!diag_on()) return;
  va_list ap;
  va_start(ap, fmt);
  t_entry = std::string(entry) + " " + vformat(fmt, ap);
  va_end(ap);
  t_note.clear();
}

void diag_note(const char *fmt, ...) {
  if (!diag_on()) return;
  va_list ap;
  va_start(ap, fmt);
  const std::string n = vformat(fmt, ap);
  va_end(ap);
  t_note += t_note.empty() ? n : " " + n;
}

void diag_launch(const void *kern, dim3 grid, dim3 block, size_t smem, int cluster, bool pdl) {
  if (!diag_on()) return;
  char geo[256];
  snprintf(geo, sizeof(geo), "grid=%u block=%u smem=%zu cluster=%d pdl=%d", grid.x * grid.y * grid.z,
           block.x * block.y * block.z, smem, cluster, pdl ? 1 : 0);
  std::string line = "mlq diag: " + (t_entry.empty() ? std::string("(internal)") : t_entry) + " -> " +
                     kernel_name(kern) + " " + geo;
  if (!t_note.empty()) line += " " + t_note;
  t_note.clear();
  static std::unordered_set<std::string> seen;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!seen.insert(line).second) return;
  fprintf(stderr, "%s\n", line.c_str());
  fflush(stderr);
}

}  // namespace mlq
