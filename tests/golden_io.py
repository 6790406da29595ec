"""Reader for the hand-written LFU trace fixtures in tests/golden/."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_lfu_trace(name):
    slots = layers = None
    inputs, events = [], []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            tok = line.split()
            if tok[0] == "slots":
                slots = int(tok[1])
            elif tok[0] == "layers":
                layers = int(tok[1])
            elif tok[0] == "in":
                inputs.append((int(tok[1]), int(tok[2]), [int(t) for t in tok[3:]]))
            elif tok[0] == "ev":
                events.append(tuple(int(t) for t in tok[1:]))
    return slots, layers, inputs, events


def lfu_trace_names():
    return sorted(n for n in os.listdir(GOLDEN) if n.startswith("lfu_") and n.endswith(".txt"))
