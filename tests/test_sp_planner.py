"""Window-aligned sequence parallelism planner (host-side, native) -- no GPU.

The planner is checked against brute force (a Python restatement of the longest-first
assignment, window sizes and ids from the oracle's window partition, send/receive counts by
counting pairs of owners), and the whole regular -> shifted -> regular cycle runs on two and
three CPU ranks over gloo: rows are moved by the plan's all-to-all, window attention is computed
locally on each rank, and the gathered result equals the single-process oracle bit for bit.
Source: [H3-fast] "Breaking the engineering bottlenecks of video-generation models", section
"Breaking the memory wall: window attention across GPUs", "Window-aligned SP".
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle


@pytest.fixture(scope="module")
def h3():
    import __graft_entry__

    __graft_entry__.build()
    import packed_varlen_attention_modality_gb300 as h3

    h3.load_library()
    return h3


GEOMS = [((32, 48, 84), (4, 8, 8), (0, 0, 0)), ((32, 48, 84), (4, 8, 8), (2, 4, 4)),
         ((6, 10, 12), (4, 8, 8), (2, 4, 4)), ((5, 7, 9), (2, 4, 4), (1, 2, 3))]


def _sizes(grid, win, shift):
    _, cu = oracle.window_partition(grid, win, shift)
    return np.diff(cu).astype(np.int64)


def _lpt(sizes, world):
    owner = np.empty(sizes.size, np.int32)
    load = np.zeros(world, np.int64)
    for i in sorted(range(sizes.size), key=lambda i: (-sizes[i], i)):
        r = int(np.argmin(load))          # first minimum: the lower rank on ties
        owner[i] = r
        load[r] += sizes[i]
    return owner, load


@pytest.mark.parametrize("grid,win,shift", GEOMS)
@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_assignment_is_longest_first_on_token_counts(h3, grid, win, shift, world):
    owner, tokens = h3.sp_assign_windows(grid, win, shift, world)
    ref_owner, ref_load = _lpt(_sizes(grid, win, shift), world)
    assert np.array_equal(owner, ref_owner) and np.array_equal(tokens, ref_load)
    assert tokens.sum() == np.prod(grid)


@pytest.mark.parametrize("world", [3, 5, 7])
def test_token_balance_beats_dealing_windows_by_count(h3, world):
    grid, win, shift = (32, 48, 84), (4, 8, 8), (2, 4, 4)   # 693 windows, cropped edges
    sizes = _sizes(grid, win, shift)
    _, tokens = h3.sp_assign_windows(grid, win, shift, world)
    by_count = [sizes[r::world].sum() for r in range(world)]
    assert tokens.max() <= max(by_count)
    assert tokens.max() - tokens.min() <= sizes.max()      # longest-first bound


@pytest.mark.parametrize("grid,win,shift", GEOMS[2:])
@pytest.mark.parametrize("world", [2, 3])
def test_layer_order_is_the_packed_order_restricted_to_the_rank(h3, grid, win, shift, world):
    owner, _ = h3.sp_assign_windows(grid, win, shift, world)
    perm, _ = oracle.window_partition(grid, win, shift)
    ids = oracle.window_ids(grid, win, shift)
    for r in range(world):
        assert np.array_equal(h3.sp_layer_order(grid, win, shift, owner, world, r),
                              perm[owner[ids[perm]] == r])


@pytest.mark.parametrize("grid,win,shift", GEOMS[2:])
@pytest.mark.parametrize("world", [2, 3])
def test_exchange_counts_and_indices_by_brute_force(h3, grid, win, shift, world):
    zero = (0, 0, 0)
    own_a, _ = h3.sp_assign_windows(grid, win, zero, world)
    own_b, _ = h3.sp_assign_windows(grid, win, shift, world)
    src = own_a[oracle.window_ids(grid, win, zero)]       # owner of every token in each layer
    dst = own_b[oracle.window_ids(grid, win, shift)]
    pairs = np.zeros((world, world), np.int64)
    np.add.at(pairs, (src, dst), 1)
    orders_a = [h3.sp_layer_order(grid, win, zero, own_a, world, r) for r in range(world)]
    orders_b = [h3.sp_layer_order(grid, win, shift, own_b, world, r) for r in range(world)]
    for r in range(world):
        p = h3.sp_exchange_plan(grid, win, zero, own_a, shift, own_b, world, r)
        assert np.array_equal(p["send_counts"], pairs[r]) and np.array_equal(p["recv_counts"], pairs[:, r])
        # what r sends to d, in order, is d's `to` order restricted to tokens r held
        sent = orders_a[r][p["send_index"]]
        off = np.concatenate([[0], np.cumsum(p["send_counts"])])
        for d in range(world):
            want = orders_b[d][src[orders_b[d]] == r]
            assert np.array_equal(sent[off[d]:off[d + 1]], want)
        # received rows land at r's `to` layout positions of those tokens
        arrived = np.concatenate([orders_b[r][src[orders_b[r]] == s] for s in range(world)])
        assert np.array_equal(orders_b[r][p["recv_position"]], arrived)


def _exchange(x_local, plan):
    """Move a rank's rows from its `from` layout to its `to` layout with the plan: gather by the
    send index, one all_to_all_single, scatter to the receive positions."""
    send = x_local.index_select(0, torch.from_numpy(plan["send_index"]).long())
    recv = torch.empty((int(plan["recv_counts"].sum()),) + tuple(x_local.shape[1:]), dtype=x_local.dtype)
    dist.all_to_all_single(recv, send, output_split_sizes=[int(c) for c in plan["recv_counts"]],
                           input_split_sizes=[int(c) for c in plan["send_counts"]])
    out = torch.empty_like(recv)
    out[torch.from_numpy(plan["recv_position"]).long()] = recv
    return out


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import packed_varlen_attention_modality_gb300 as h3

    grid, win, shift, zero = (6, 10, 12), (4, 8, 8), (2, 4, 4), (0, 0, 0)
    n, H, D = 720, 2, 8
    x = torch.from_numpy(np.random.default_rng(31).standard_normal((n, H, D)))    # same on every rank
    own_a, _ = h3.sp_assign_windows(grid, win, zero, world)
    own_b, _ = h3.sp_assign_windows(grid, win, shift, world)
    order_a = h3.sp_layer_order(grid, win, zero, own_a, world, rank)
    order_b = h3.sp_layer_order(grid, win, shift, own_b, world, rank)
    local_a = x[torch.from_numpy(order_a).long()].contiguous()
    local_b = _exchange(local_a, h3.sp_exchange_plan(grid, win, zero, own_a, shift, own_b, world, rank))
    ok_move = bool(torch.equal(local_b, x[torch.from_numpy(order_b).long()]))
    # shifted-window attention on this rank's windows only (q = k = v = the moved rows)
    sizes = np.diff(oracle.window_partition(grid, win, shift)[1])
    mine = sizes[own_b == rank]
    cu = np.concatenate([[0], np.cumsum(mine)])
    lb = local_b.numpy()                                    # fp64 (a torch tensor would pass through fp32)
    o_local, _ = oracle.varlen_attention(lb, lb, lb, cu)
    full = torch.zeros((n, H, D), dtype=torch.float64)
    full[torch.from_numpy(order_b).long()] = torch.from_numpy(o_local)
    dist.all_reduce(full)                                   # each token is written by one rank
    # and back to the regular layout
    back = _exchange(local_b, h3.sp_exchange_plan(grid, win, shift, own_b, zero, own_a, world, rank))
    ok_back = bool(torch.equal(back, local_a))
    q.put((rank, ok_move, ok_back, full.numpy()))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_regular_shifted_regular_cycle_on_cpu_ranks(h3, world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=300) for _ in range(world)]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    grid, win, shift = (6, 10, 12), (4, 8, 8), (2, 4, 4)
    x = np.random.default_rng(31).standard_normal((720, 2, 8))
    perm, cu = oracle.window_partition(grid, win, shift)
    xp = oracle.window_pack(x, perm)
    ref, _ = oracle.varlen_attention(xp, xp, xp, cu)
    ref = oracle.window_unpack(ref, perm)
    for rank, ok_move, ok_back, full in res:
        assert ok_move and ok_back, rank
        assert np.array_equal(full, ref), rank
