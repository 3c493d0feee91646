"""Plain-Python oracle of the tiered store's admission policy (LFRU).

TEST INFRASTRUCTURE ONLY (see the package docstring): the library never
imports it.  It follows "Colibrì 深度解析" §三 as written there:

  - every expert keeps a heat (route counts with exponential decay) and the
    tick of its last route;
  - LFRU score = heat * 256 + recent, recent = 255 - age for an age below 255
    ticks, else 0: frequency is the primary signal, and a recent access is
    worth at most 255 points against 256 for one count;
  - an expert is promoted over a colder one only if hot > cold + cold / 4 + 4,
    computed in a wider integer so that a saturated counter cannot wrap the
    threshold (hysteresis against ping-pong).

Readings where the page is silent (listed in the design notes): the decay is
heat - heat // 8 per tick before the tick's counts are added, saturating at
2**32 - 1; candidates are the routed experts used in the tick that are not
resident, best score first (ties: lower id); a candidate takes the lowest
free slot (cold = 0) or else the resident routed expert of lowest score (ties:
lowest slot); experts considered in a tick (admitted or not) are neither
reconsidered nor evicted in that tick; shared experts are never moved.
"""

U32 = 2 ** 32


def recent(clock, last):
    age = (clock - last) % U32
    return 255 - age if age < 255 else 0


def score(heat, last, clock):
    return heat * 256 + recent(clock, last)


def should_promote(hot, cold):
    return hot > cold + cold // 4 + 4


class TierState:
    def __init__(self, n_experts, n_shared, owners):
        self.E, self.S = n_experts, n_shared
        self.owner = list(owners)
        self.slot_of = [-1] * (n_experts + n_shared)
        for sl, e in enumerate(self.owner):
            if e >= 0:
                self.slot_of[e] = sl
        self.heat = [0] * n_experts
        self.last = [0] * n_experts
        self.clock = 0

    def tick(self, counts, max_uploads):
        """One policy tick from the call's route counts [E]; returns the
        (expert, slot) uploads in order."""
        E = self.E
        self.clock = (self.clock + 1) % U32
        for e in range(E):
            h = self.heat[e]
            self.heat[e] = min(h - (h >> 3) + int(counts[e]), U32 - 1)
            if counts[e]:
                self.last[e] = self.clock
        considered, uploads = set(), []
        while len(uploads) < max_uploads:
            cands = [e for e in range(E)
                     if counts[e] and self.slot_of[e] < 0 and e not in considered]
            if not cands:
                break
            c = min(cands, key=lambda e: (-score(self.heat[e], self.last[e], self.clock), e))
            free = [sl for sl, o in enumerate(self.owner) if o < 0]
            target, cold = None, 0
            if free:
                target = min(free)
            else:
                res = [sl for sl, o in enumerate(self.owner) if 0 <= o < E and o not in considered]
                if res:
                    target = min(res, key=lambda sl: (score(self.heat[self.owner[sl]],
                                                            self.last[self.owner[sl]],
                                                            self.clock), sl))
                    cold = self.heat[self.owner[target]]
            if target is not None and should_promote(self.heat[c], cold):
                old = self.owner[target]
                if old >= 0:
                    self.slot_of[old] = -1
                self.owner[target] = c
                self.slot_of[c] = target
                uploads.append((c, target))
            considered.add(c)
        return uploads
