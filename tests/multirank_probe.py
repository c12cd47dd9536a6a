"""Run under torchrun with gloo on the CPU: exercises bench.py's multi-rank plumbing."""
import json
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

rank, world, local = bench.dist_env()
dist = bench.init_dist(world, "gloo")
times = [1.0 + rank, 10.0 * (rank + 1), 0.5]
mx = bench.max_over_ranks(dist, times)
bench.barrier(dist)
value = bench.whole_job_throughput(8192, world, mx[0])
# one write per line: both ranks share the pipe, and print() may issue the text
# and its newline as two writes when stdout is unbuffered
sys.stdout.write(json.dumps({"rank": rank, "world": world, "local": local, "max": mx, "value": value}) + "\n")
sys.stdout.flush()
dist.destroy_process_group()
