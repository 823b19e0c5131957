// Host NUMA placement of the pinned KV caches.
//
// DirectKV's KV Cache Manager keeps the offloaded cache in the CPU memory the
// GPU reaches over its own host link ("Paper Notes: DirectKV", System
// Architecture, KV Cache Manager).  On a machine with several NUMA nodes a
// replica's pinned pages should sit on the node attached to its GPU, or every
// zero-copy read crosses the CPU-to-CPU fabric as well.  This file finds that
// node (the GPU's PCI device's numa_node in sysfs) and sets the calling
// thread's memory policy to prefer it while the caches are allocated and
// pinned; the policy in force before is restored afterwards.  Host code only,
// no libnuma: the two policy system calls are made directly.
#include <ctype.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <sys/mman.h>
#include <sys/syscall.h>
#include <unistd.h>

#include <cuda_runtime.h>

#include "numa_host.h"

namespace dkv {
namespace {

constexpr int kMpolDefault = 0;
constexpr int kMpolPreferred = 1;
constexpr int kMpolFNode = 1;     // get_mempolicy: return a node id
constexpr int kMpolFAddr = 2;     // get_mempolicy: of the page at addr
constexpr int kMaskWords = 16;    // node masks of 1024 bits
constexpr unsigned long kMaxNode = kMaskWords * 64 + 1;  // the kernel reads maxnode - 1 bits

long get_policy(int* mode, unsigned long* mask) {
  return syscall(SYS_get_mempolicy, mode, mask, kMaxNode, nullptr, 0);
}
long set_policy(int mode, const unsigned long* mask) {
  return syscall(SYS_set_mempolicy, mode, mode == kMpolDefault ? nullptr : mask,
                 mode == kMpolDefault ? 0 : kMaxNode);
}

}  // namespace

int pci_numa_node(const char* bus_id, const char* sysfs_root) {
  if (!bus_id) return -1;
  unsigned dom = 0, bus = 0, devno = 0, fn = 0;
  if (sscanf(bus_id, "%x:%x:%x.%x", &dom, &bus, &devno, &fn) != 4) return -1;
  char path[512];
  snprintf(path, sizeof path, "%s/bus/pci/devices/%04x:%02x:%02x.%x/numa_node",
           sysfs_root && *sysfs_root ? sysfs_root : "/sys", dom, bus, devno, fn);
  FILE* f = fopen(path, "r");
  if (!f) return -1;
  char buf[32] = {0};
  const size_t n = fread(buf, 1, sizeof buf - 1, f);
  fclose(f);
  if (n == 0) return -1;
  char* end = nullptr;
  const long v = strtol(buf, &end, 10);
  if (end == buf) return -1;
  while (*end && isspace((unsigned char)*end)) ++end;
  if (*end || v < 0 || v >= kMaskWords * 64) return -1;
  return (int)v;
}

int device_numa_node(int device) {
  const char* off = getenv("DKV_NUMA");
  if (off && strcmp(off, "0") == 0) return -1;
  char bus_id[64];
  if (cudaDeviceGetPCIBusId(bus_id, sizeof bus_id, device) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  return pci_numa_node(bus_id, nullptr);
}

int page_numa_node(const void* p) {
  int node = -1;
  if (!p) return -1;
  if (syscall(SYS_get_mempolicy, &node, nullptr, 0, const_cast<void*>(p),
              kMpolFNode | kMpolFAddr) != 0)
    return -1;
  return node;
}

NumaScope::NumaScope(int node) : active_(false), mode_(kMpolDefault) {
  memset(mask_, 0, sizeof mask_);
  if (node < 0 || node >= kMaskWords * 64) return;
  if (get_policy(&mode_, mask_) != 0) return;
  unsigned long want[kMaskWords] = {0};
  want[node / 64] = 1ul << (node % 64);
  active_ = set_policy(kMpolPreferred, want) == 0;
}

NumaScope::~NumaScope() {
  if (active_) set_policy(mode_, mask_);
}

}  // namespace dkv

// The NUMA node sysfs gives for a PCI device (bus id as cudaDeviceGetPCIBusId
// prints it), -1 if unknown.  sysfs_root: null or "" for /sys.
extern "C" int dkv_pci_numa_node(const char* pci_bus_id, const char* sysfs_root) {
  return dkv::pci_numa_node(pci_bus_id, sysfs_root);
}

// Places one page with the calling thread's policy preferring `node` (as the
// cache allocation does) and reports the node it landed on, or -1.
extern "C" int dkv_numa_probe(int node) {
  const long page = sysconf(_SC_PAGESIZE);
  int placed = -1;
  {
    dkv::NumaScope scope(node);
    void* p = mmap(nullptr, (size_t)page, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS,
                   -1, 0);
    if (p == MAP_FAILED) return -1;
    memset(p, 1, (size_t)page);  // first touch: the page is allocated here
    placed = dkv::page_numa_node(p);
    munmap(p, (size_t)page);
  }
  return placed;
}
