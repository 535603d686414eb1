"""Host logic of bench.py: replica aggregation over torch.distributed (gloo,
world size 2, CPU) and the workload accounting."""
import os
import socket

import torch.multiprocessing as mp

import bench
import synth


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    units, secs = bench.aggregate(100.0 * (rank + 1), 0.5 + rank)
    q.put((rank, units, secs))
    dist.destroy_process_group()


def test_aggregate_sums_units_and_takes_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for _, units, secs in res:
        assert units == 300.0 and secs == 1.5


def test_single_process_aggregate_is_identity():
    assert bench.aggregate(5.0, 2.0) == (5.0, 2.0)


def test_workload_accounting():
    cfg = bench.config_dict()
    assert cfg["workload"] == "gpt2_small_mlp_backward"
    wl = synth.WORKLOADS["mlp"]
    assert cfg["flops_per_step"] == sum(4 * l.BT * l.C * l.OC + l.BT * l.OC for l in wl.layers)
    assert sum(bench.layer_bytes(l) for l in wl.layers) * bench.N_SETS > 129e6 * 2


def test_traffic_is_null_for_a_changed_kernel(tmp_path, monkeypatch):
    # a summary taken on another kernel source must not be reported
    assert bench.kernel_source_sha() and len(bench.kernel_source_sha()) == 12
    prof = os.path.join(bench.ROOT, "profiles", "tc_mmbwd_kernel_mlp.md")
    if os.path.exists(prof):
        t = bench.profiled_traffic()
        assert t is None or t > 0


class _FakeEvent:
    """Stands in for torch.cuda.Event: elapsed time is fixed; `query` says
    whether the spin in front of it has ended, by a script of answers."""

    def __init__(self, log, answers=None, **kw):
        self.log, self.answers = log, answers

    def record(self, stream=None):
        self.log.append("record")

    def query(self):
        return self.answers.pop(0)

    def synchronize(self):
        pass

    def elapsed_time(self, other):
        return 2.0  # ms


class _FakeCuda:
    def __init__(self, answers):
        self.log, self.answers, self.spins = [], answers, []

    def Event(self, **kw):
        return _FakeEvent(self.log, self.answers)

    def _sleep(self, cycles):
        self.spins.append(cycles)
        self.log.append("spin")

    def stream(self, s):
        import contextlib

        return contextlib.nullcontext()

    def synchronize(self):
        pass


class _FakeTorch:
    def __init__(self, answers):
        self.cuda = _FakeCuda(answers)


def test_time_back_to_back_queues_each_batch_behind_a_spin():
    # first batch: the spin ended before the batch was queued (query True), so
    # the batch is taken again behind a spin twice as long; then it held
    ft = _FakeTorch([True, False, False])
    calls = []
    sec = bench.time_back_to_back(ft, None, [lambda: calls.append(1)], per_batch=4, batches=2)
    assert sec == 2.0e-3 / 4
    assert len(ft.cuda.spins) == 3
    assert abs(ft.cuda.spins[1] - 2 * ft.cuda.spins[0]) <= 2 and ft.cuda.spins[2] == ft.cuda.spins[1]
    assert ft.cuda.spins[0] >= 50 * bench.SPIN_CYCLES_PER_US
    assert len(calls) == 2 + 3 * 4  # warm-up (each call twice) and three queued batches
    # every batch's first event comes after its spin's event
    assert ft.cuda.log[-4:] == ["spin", "record", "record", "record"]


def test_code_hash_ignores_comments_and_layout_only(tmp_path):
    # the profiles' kernel_source_sha: edits of comments or white space keep it,
    # any change of code (a string literal included) does not
    import ncu_harness as H

    def sha(name, text):
        p = tmp_path / name
        p.write_text(text)
        return H.code_sha([p])

    base = sha("a.cu", 'int f(int x) { return x + 1; }  // one\n/* two */\nconst char* s = "a // b";\n')
    relaid = sha("b.cu", '// header\nint f(int x) {\n    return x + 1;   // other words\n}\n'
                         '/* several\n   lines */ const char* s = "a // b";\n')
    code = sha("c.cu", 'int f(int x) { return x + 2; }\nconst char* s = "a // b";\n')
    literal = sha("d.cu", 'int f(int x) { return x + 1; }\nconst char* s = "a ";\n')
    assert base == relaid
    assert len({base, code, literal}) == 3
    assert bench.kernel_source_sha() == H.source_sha(("tc_gemm.cu", "ptx.cuh", "internal.h"))
