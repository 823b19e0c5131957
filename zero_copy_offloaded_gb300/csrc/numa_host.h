// Host NUMA placement of the pinned caches (host code only).
#pragma once

namespace dkv {

// NUMA node of the PCI device with this bus id ("0000:1b:00.0"), read from
// <sysfs_root>/bus/pci/devices/<id>/numa_node (sysfs_root null: /sys); -1 when
// unknown, absent or malformed.
int pci_numa_node(const char* bus_id, const char* sysfs_root);

// The node attached to CUDA device `device`, -1 if unknown or if DKV_NUMA=0.
int device_numa_node(int device);

// Node holding the (already touched) page at p, -1 if unknown.
int page_numa_node(const void* p);

// While alive, the calling thread's memory policy prefers `node` (pages it
// touches or pins come from that node when it has room); the policy in force
// before is restored on destruction.  A negative node changes nothing.
class NumaScope {
 public:
  explicit NumaScope(int node);
  ~NumaScope();
  NumaScope(const NumaScope&) = delete;
  NumaScope& operator=(const NumaScope&) = delete;

 private:
  bool active_;
  int mode_;
  unsigned long mask_[16];
};

}  // namespace dkv
