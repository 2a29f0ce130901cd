"""Worker for the two-rank CPU tests (spawned processes import it by name)."""
import os
import sys


def max_over_ranks(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    r, w, _ = bench.init_dist(None)
    bench.barrier(w)
    got = bench.allreduce_max(1.5 + r, w, "cpu")
    bench.barrier(w)
    with open(os.path.join(out_dir, f"rank{r}.txt"), "w") as f:
        f.write(f"{r} {w} {got}\n")
    bench._PG.destroy_process_group()
