"""One rank of the world-size-2 CPU test of bench.py's multi-rank host logic.

Launched by tests/test_ranks_cpu.py through torch.distributed.run (the way
bench.py is launched for N > 1) with the gloo backend on 127.0.0.1.  Each
rank reports a different time; the job's time is the slowest rank's.  Each
rank writes its result to RANK_OUT_DIR/rank<r>.json.
"""
import json
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def main():
    world = int(os.environ["WORLD_SIZE"])
    rank = int(os.environ["RANK"])
    torch.distributed.init_process_group("gloo")
    dev = torch.device("cpu")
    mine = 2.5 + 5.0 * rank
    slowest = bench.max_over_ranks(mine, world, dev)
    torch.distributed.barrier()
    out = os.path.join(os.environ["RANK_OUT_DIR"], f"rank{rank}.json")
    with open(out, "w") as f:
        json.dump({"rank": rank, "world": world, "mine": mine, "slowest": slowest}, f)
    torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
