"""GPU tests of the streamed-expert cache paths through the C ABI.

Devtrends page "Como executar um modelo de 26 bilhoes de parametros em dois
gigabytes de memoria em um Mac comum", section "Qual e o principal truque da
arquitetura": per token and layer the router picks 8 experts, a 16-slot LFU
cache is checked and missing experts are read from slower memory while the
shared-expert branch runs. Two ways to run it are checked here against the
CPU oracle's LFU simulator (oracle.LFU) and against the resident path:

  - the LFU metadata on the device (tf_layer_step_device_cache): a one-warp
    kernel decides hits and victims, a copy kernel fetches the misses from the
    pinned host store; the trace and the slot contents must equal the oracle's
    event for event, and every layer output must equal the resident path's bit
    for bit;
  - the host metadata with the miss fills striped over several copy streams
    (tf_expert_cache_set_copy_streams), at 8 and 32 slots per layer;
  - chunked prefill through the cache (tf_layer_prefill_cached): a chunk's
    experts stream through the slots in waves, each loaded expert serving all
    of the chunk's rows that need it.

The router logits carry the streaming workload's bias (Zipf popularity,
per-step noise, a repeat of the previous step's experts), so that steps mix
hits, cold fills and evictions.
"""
import numpy as np
import pytest
import torch

import bit_expert_streaming_layer_b300 as B
import oracle as O
import workload as W
from workload.model import SyntheticStack, hidden_tensor

pytestmark = pytest.mark.gpu
DEV = "cuda"
SMALL = dict(H=320, I=192, E=24, k=4, S=128)
FULL = dict(H=2816, I=704, E=128, k=8, S=2112)


def nan_bf16(n):
    return torch.full((n,), float("nan"), dtype=torch.bfloat16, device=DEV)


def _bias(seed, l, E, prev_ids, step, alpha=0.1, sigma=1.5):
    b = W.zipf_bias(seed, l, E, 1.1, alpha)[0] + W.route_noise(seed, l, step, E, sigma)
    if prev_ids is not None and W.coin(seed, l, step):
        b = b.copy()
        b[prev_ids] += 30.0
    return b.astype(np.float32)


def _device_cache(stack, n_slots, trace_cap):
    pool = torch.zeros(stack.L * n_slots * stack.slot, dtype=torch.uint8, device=DEV)
    state = torch.zeros(B.tf_device_cache_state_bytes(stack.L, n_slots, stack.E, trace_cap), dtype=torch.uint8,
                        device=DEV)
    return B.DeviceCache(stack.L, n_slots, stack.E, stack.slot, pool, stack.store, state, trace_cap)


def _run(cfg, L, slots, steps, seed, mode, n_streams=1):
    """Run `steps` tokens through L layers on the cached path (mode 'device' or 'host') and the resident
    path side by side, fresh inputs per step; returns (trace, oracle trace, stats list, cache handle)."""
    H, E, k = cfg["H"], cfg["E"], cfg["k"]
    cached = SyntheticStack(seed, L, resident=False, n_slots=slots, **cfg)
    resident = SyntheticStack(seed, L, resident=True, **cfg)
    fetch = torch.cuda.Stream(priority=-1)
    streams = [torch.cuda.Stream() for _ in range(n_streams)]
    dcache = _device_cache(cached, slots, L * steps * k) if mode == "device" else None
    if mode == "host" and n_streams > 1:
        cached.cache.set_copy_streams(streams)
    lfu = O.LFU(L, slots)
    want, stats = [], []
    prev = [None] * L
    bias_d = torch.empty(E, dtype=torch.float32, device=DEV)
    for step in range(steps):
        cur_c = hidden_tensor(seed, step, 1, H)[0]
        cur_r = cur_c.clone()
        for l in range(L):
            bias_d.copy_(torch.from_numpy(_bias(seed, l, E, prev[l], step)))
            out_c, out_r = nan_bf16(H), nan_bf16(H)
            measure = 1 if (step + l) % 3 == 0 else 0
            if mode == "device":
                st = B.tf_layer_step_device_cache(cached.layers[l], dcache, l, cur_c, out_c, bias_d, 0, None, fetch,
                                                  measure)
            else:
                st = B.tf_layer_step(cached.layers[l], cached.cache, l, step, cached.store, cur_c, out_c, 1, bias_d,
                                     0, None, streams[0], measure)
            B.tf_layer_step(resident.layers[l], None, l, step, None, cur_r, out_r, 1, bias_d, 0)
            torch.cuda.synchronize()
            ids = cached.layers[l].routing_tensors()[0][0].cpu().numpy()
            prev[l] = ids
            ev = lfu.step(step, l, ids)
            want += ev
            if measure or mode == "host":
                assert st.hits + st.misses == k and st.misses == sum(1 for e in ev if not e[3])
                assert list(st.ids[:k]) == ids.tolist()
                assert st.bytes_fetched == st.misses * cached.payload
                stats.append(st)
            # the cached path computes the same bits as the resident one
            assert torch.equal(out_c.view(torch.int16), out_r.view(torch.int16)), (step, l)
            cur_c, cur_r = out_c, out_r
    trace = dcache.trace() if mode == "device" else cached.cache.trace()
    for l in range(L):   # the slot contents at the end, as the oracle has them
        got = dcache.state(l) if mode == "device" else cached.cache.state(l)
        exp = lfu.state(l)
        assert all(np.array_equal(a, b) for a, b in zip(got, exp)), l
    if mode == "device":
        hits, misses, events = dcache.counters()
        assert events == len(want) and hits == sum(e[3] for e in want) and misses == len(want) - hits
        dcache.close()
    cached.close()
    resident.close()
    return trace, want, stats


@pytest.mark.parametrize("cfg,L,slots,steps", [
    (SMALL, 3, 6, 20), (FULL, 3, 16, 10), (FULL, 2, 8, 8), (FULL, 2, 32, 8)],
    ids=["small_6", "full_16", "full_8", "full_32"])
def test_device_cache_trace_state_and_outputs(cfg, L, slots, steps):
    trace, want, _ = _run(cfg, L, slots, steps, 52, "device")
    assert trace == want
    assert any(not e[3] and e[5] >= 0 for e in want)   # evictions happened
    assert any(e[3] for e in want)                       # and hits


@pytest.mark.parametrize("slots,n_streams", [(8, 2), (32, 3), (16, 4)], ids=["8_slots_2", "32_slots_3", "16_slots_4"])
def test_host_cache_striped_copy_streams(slots, n_streams):
    trace, want, stats = _run(FULL, 2, slots, 6, 53, "host", n_streams)
    assert trace == want
    assert any(s.misses >= 2 for s in stats)    # steps whose fills really were spread over streams
    assert all(s.copy_ms >= 0.0 and s.stall_ms >= 0.0 for s in stats)


def test_device_cache_rejects_bad_arguments():
    cfg = SMALL
    st = SyntheticStack(54, 1, resident=False, n_slots=6, **cfg)
    state = torch.zeros(B.tf_device_cache_state_bytes(1, 6, cfg["E"], 16), dtype=torch.uint8, device=DEV)
    pool = torch.zeros(6 * st.slot, dtype=torch.uint8, device=DEV)
    with pytest.raises(B.TFError) as e:      # state too small
        B.DeviceCache(1, 6, cfg["E"], st.slot, pool, st.store, state[:1024], 16)
    assert e.value.status == B.TF_ERR_INVALID_ARG
    with pytest.raises(B.TFError) as e:      # more slots than the LFU kernel holds
        B.DeviceCache(1, 2048, cfg["E"], st.slot, pool, st.store, state, 16)
    assert e.value.status == B.TF_ERR_INVALID_ARG
    pageable = torch.zeros(cfg["E"] * st.slot, dtype=torch.uint8)     # not pinned: not mapped for the device
    with pytest.raises(B.TFError) as e:
        B.DeviceCache(1, 6, cfg["E"], st.slot, pool, pageable, state, 16)
    assert e.value.status == B.TF_ERR_NOT_SUPPORTED
    c = B.DeviceCache(1, 6, cfg["E"], st.slot, pool, st.store, state, 16)
    x = hidden_tensor(54, 0, 1, cfg["H"])[0]
    with pytest.raises(B.TFError) as e:      # a layer index beyond the cache
        B.tf_layer_step_device_cache(st.layers[0], c, 1, x, nan_bf16(cfg["H"]), None, 0, None,
                                     torch.cuda.Stream())
    assert e.value.status == B.TF_ERR_INVALID_ARG
    c.close()
    st.close()


# ------------------------------------------------------------- chunked prefill through the cache

def _waves(ids, n_slots):
    """The chunk's distinct experts in order of first use (token order, then rank), cut into waves of n_slots."""
    order = []
    for e in ids.reshape(-1).tolist():
        if e not in order:
            order.append(e)
    return [np.array(order[i:i + n_slots], np.int32) for i in range(0, len(order), n_slots)]


@pytest.mark.parametrize("cfg,L,slots,T,chunks", [
    (dict(H=512, I=256, E=24, k=4, S=128), 2, 6, 40, 3),
    (FULL, 1, 16, 128, 2)], ids=["small", "full"])
def test_chunked_prefill_through_the_cache(cfg, L, slots, T, chunks):
    """Devtrends page, section "Desempenho no mundo real": prefill in chunks, one loaded expert serving all of the
    chunk's rows. Every layer output equals the resident batched step's bit for bit; the LFU trace and the slots
    equal the oracle's fed the same waves (each wave one step, its experts in order)."""
    H, E, k = cfg["H"], cfg["E"], cfg["k"]
    seed = 57
    cached = SyntheticStack(seed, L, resident=False, n_slots=slots, T_max=T, **cfg)
    resident = SyntheticStack(seed, L, resident=True, T_max=T, **cfg)
    cs = torch.cuda.Stream()
    lfu = O.LFU(L, slots)
    want = []
    step = [0] * L
    for c in range(chunks):
        x = hidden_tensor(seed, c, T, H)
        cur_c, cur_r = x, x.clone()
        for l in range(L):
            out_c = torch.full_like(x, float("nan"))
            out_r = torch.full_like(x, float("nan"))
            st = B.tf_layer_prefill_cached(cached.layers[l], cached.cache, l, step[l], cached.store, cur_c, out_c, T,
                                           None, 0, None, cs)
            B.tf_layer_step(resident.layers[l], None, l, 0, None, cur_r, out_r, T)
            torch.cuda.synchronize()
            ids = cached.layers[l].routing_tensors(T)[0].cpu().numpy()
            waves = _waves(ids, slots)
            assert st.waves == len(waves)
            ev = []
            for w, wave in enumerate(waves):
                ev += lfu.step(step[l] + w, l, wave)
            want += ev
            assert st.misses == sum(1 for e in ev if not e[3]) and st.hits + st.misses == len(ev)
            assert st.bytes_fetched == st.misses * cached.payload
            step[l] += st.waves
            assert torch.equal(out_c.view(torch.int16), out_r.view(torch.int16)), (c, l)
            cur_c, cur_r = out_c, out_r
    assert cached.cache.trace() == want
    for l in range(L):
        got, exp = cached.cache.state(l), lfu.state(l)
        assert all(np.array_equal(a, b) for a, b in zip(got, exp)), l
    assert any(not e[3] and e[5] >= 0 for e in want)       # evictions inside chunks
    cached.close()
    resident.close()


def test_chunked_prefill_copy_failure_rolls_back():
    cfg = dict(H=512, I=256, E=24, k=4, S=128)
    st = SyntheticStack(58, 1, resident=False, n_slots=6, T_max=16, **cfg)
    cs = torch.cuda.Stream()
    x = hidden_tensor(58, 0, 16, cfg["H"])
    out = torch.empty_like(x)
    B.tf_test_fail_nth_copy(2)            # the first wave's second copy fails
    with pytest.raises(B.TFError) as e:
        B.tf_layer_prefill_cached(st.layers[0], st.cache, 0, 0, st.store, x, out, 16, None, 0, None, cs)
    B.tf_test_fail_nth_copy(0)
    assert e.value.status == B.TF_ERR_CUDA and "rolled back" in str(e.value)
    torch.cuda.synchronize()
    ex, cnt, lu = st.cache.state(0)
    assert (ex >= 0).sum() == 0
    s2 = B.tf_layer_prefill_cached(st.layers[0], st.cache, 0, 1, st.store, x, out, 16, None, 0, None, cs)
    torch.cuda.synchronize()
    assert s2.waves >= 1 and not torch.isnan(out.float()).any()
    st.close()

