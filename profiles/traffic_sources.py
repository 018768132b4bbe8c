"""Record the DRAM traffic of one ncu capture in profiles/ncu_traffic.json.

    python profiles/traffic_sources.py <workload> <kernel> <dram_bytes_per_launch> <command...>

Stores the bytes with the sha256 of the kernel's source files, so bench.py
reports the figure only while the kernel is unchanged."""
import hashlib
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SOURCES = {
    "ffn_tc_kernel<0>": ["mixture_experts_ffn_19_b300/csrc/ffn_tc.cu",
                         "mixture_experts_ffn_19_b300/csrc/common.cuh"],
}


def main(workload, kernel, nbytes, *command):
    srcs = SOURCES[kernel]
    h = hashlib.sha256()
    for s in srcs:
        with open(os.path.join(ROOT, s), "rb") as f:
            h.update(f.read())
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    data = json.load(open(path)) if os.path.exists(path) else {}
    data.setdefault(workload, {})[kernel] = {
        "dram_bytes_per_launch": float(nbytes), "sources": srcs,
        "source_sha256": h.hexdigest(), "command": " ".join(command)}
    with open(path, "w") as f:
        json.dump(data, f, indent=1, sort_keys=True)


if __name__ == "__main__":
    main(*sys.argv[1:])
